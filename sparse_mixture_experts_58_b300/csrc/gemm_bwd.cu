// Backward of the grouped expert GEMMs (gradients for training) on CTA pairs.
//
// The forward of one expert on its rows X (tokens as rows):
//   U = X W1^T,  V = X W3^T,  H = silu(U) * V,  Y = H W2^T,  out[t] += g Y[row].
// With G the upstream gradient of the layer output gathered to the rows
// (G[row] = dout[t]) and g the row's gate, the chain rule gives
//   Z  = G W2                          dH = g Z
//   dU = dH * V * silu'(U)             dV = dH * silu(U)
//   dg[row] = sum_c H[row][c] Z[row][c]            (<dout, y>, for the router)
//   dX = dU W1 + dV W3
//   dW1 = dU^T X,  dW3 = dV^T X,  dW2 = G^T (g H)
// (Mixtral's experts are SwiGLU networks with their own weights: "Mixtral of
// Experts" (azimuth.plus), expert paragraph; the layer output is the gate-
// weighted sum: "Mixtral & Sparse MoE (2024) > The Solution", routing
// paragraph.)
//
// Four modes of one kernel, all on CTA pairs (tcgen05 .cta_group::2, M = 256
// rows of the weight side, 128 in each CTA, as in gemm_pair.cu):
//   kUV  U and V again (recomputed, not kept from the forward): A = W1/W3
//        rows (K-major), B = token rows; stores U and V (bf16).
//   kZ   Z = G W2: A = W2 read MN-major (its rows are the contraction);
//        epilogue forms dU, dV, g H (bf16) and per-row partial sums of
//        H * Z over 32-feature blocks.
//   kDX  dX = dU W1 + dV W3: A = W1 then W3 read MN-major, B = dU then dV;
//        fp32 rows.
//   kWG  weight gradients: A and B both activations read MN-major, the
//        contraction runs over one expert's rows; fp32 [M][N] per expert.
// Rows are grouped by expert with each expert's block starting on a multiple
// of 64 and padded with zero rows, so a 64-row contraction step never mixes
// experts.
//
// MN-major operand tiles are TMA boxes of 64 contraction rows x 64 elements
// (128 bytes, 128-byte swizzle); a 128-wide tile is two boxes 8 KB apart.
// The matrix descriptor names that layout: the 64-element chunks along M (or
// N) LBO = 8 KB apart, groups of 8 contraction rows SBO = 1 KB apart, and a
// 16-deep MMA step advances the start by 16 rows (2 KB).
//
// Roles as in gemm_pair.cu (warp 0 TMA, warp 1 MMA), but with eight
// epilogue warps: the two warps on each tensor-memory lane quarter take
// alternate 32-column chunks, since the kZ and kWG epilogues do more work per
// element than one warp per quarter hides behind the MMAs.  Five 32 KB ring
// stages leave room for the kWG transpose tiles.  Barriers and bounded waits as
// in gemm_pair.cu (an accumulator is released by all 16 epilogue warps of the
// pair).
#include <string.h>

#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kPairM = 256;
constexpr int kHalfM = 128;
constexpr int kMaxTok = 256;
constexpr int kTokMaps = kMaxTok / 16;
constexpr int kStages = 5;
constexpr int kMaxE = MOE_MAX_EXPERTS;
constexpr int kEpiWarps = 8;  // two per tensor-memory lane quarter
// a warp's 32-column chunks of an accumulator are kChunkStep apart
constexpr int kChunkStep = 32 * (kEpiWarps / 4);
static_assert(kEpiWarps % 4 == 0, "whole lane quarters per epilogue warp set");
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kBox = 64 * 128;              // one 64 x 64 bf16 box
constexpr int kABytes = 2 * kBox;           // 128 weight-side rows x 64, or 64 x 128 MN-major
constexpr int kBBytes = 2 * kBox;           // this CTA's half of the token / N side
constexpr int kRing = kStages * (kABytes + kBBytes);
constexpr int kBars = (2 * kStages + 6) * 8;
constexpr int kMisc = 16 + 4 * (4 * kMaxE + 2);
constexpr int kXpitch = 36;              // floats per row of the transpose tile (16-byte rows)
constexpr int kXpose = kEpiWarps * 32 * kXpitch * 4;  // kWG: a 32 x 32 fp32 tile per epilogue warp
constexpr size_t kSmem = 1024 + kRing + kXpose + kBars + kMisc;
constexpr uint32_t kAccCols = kMaxTok;
constexpr uint32_t kTmemCols = 2 * kAccCols;
constexpr int kAccEmptyArrivals = 2 * kEpiWarps;  // lane 0 of each epilogue warp, both CTAs
constexpr uint16_t kBothCtas = 0x3;

enum Mode { kUV = 0, kZ = 1, kDX = 2, kWG = 3 };

// Matrix descriptor of an MN-major operand tile (layout above).
__device__ __forceinline__ uint64_t desc_mnmajor_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((kBox >> 4) & 0x3FFF) << 16;  // LBO: next 64 along M/N
    d |= static_cast<uint64_t>(1024u >> 4) << 32;            // SBO: next 8 contraction rows
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

// Instruction descriptor with A and/or B MN-major (bits 15 and 16).
__host__ __device__ constexpr uint32_t idesc_major(int M, int N, bool a_mn, bool b_mn) {
    return ptx::idesc_bf16_f32(M, N) | (a_mn ? (1u << 15) : 0u) | (b_mn ? (1u << 16) : 0u);
}

struct BwdArgs {
    CUtensorMap tok0[kTokMaps];  // token rows, K-major, box {64, 8 (i + 1)}: X (kUV), G (kZ), dU (kDX)
    CUtensorMap tok1[kTokMaps];  // dV (kDX)
    CUtensorMap w0[kMaxE];       // box {64, 64}: W1 (kUV, kDX), W2 (kZ)
    CUtensorMap w1[kMaxE];       // box {64, 64}: W3 (kUV, kDX)
    CUtensorMap act_a[3];        // kWG, box {64, 64}: dU, dV, G  ([rows][M])
    CUtensorMap act_b[3];        // kWG, box {64, 64}: X, X, gH   ([rows][N])
    const int *offsets;          // [E + 1] row offsets, multiples of 64
    __nv_bfloat16 *U, *V;        // kUV out, kZ in: feature-major [ffn][rows]
    __nv_bfloat16 *dU, *dV, *gH; // kZ out: [rows][ffn]
    const float *row_gate;       // kZ: [rows] gate of each row (0 for padding)
    float *dgp;                  // kZ: [rows][ffn / 32]
    float *dx_rows;              // kDX: [rows][d]
    float *wgrad[3][kMaxE];      // kWG: per gradient and expert, [M][N] fp32
    int wg_M[3], wg_N[3];        // kWG: gradient shapes
    int wg_count;                // kWG: gradients in this launch
    int *status;
    unsigned long long wait_limit_ns;
    int E, rows, d, ffn;
};

struct BUnit {
    int e, t0, nvalid, ntok;  // token modes: expert and token tile
    int n0;                   // first weight-side feature (token modes) or M row (kWG)
    int kb0, kb1;             // contraction blocks
    int g, m0, nw0;           // kWG: gradient, M and N tile starts
};

template <int MODE>
__device__ __forceinline__ BUnit decode_bwd_unit(int u, const int *s_off, const int *s_ntt,
                                                 const int *s_nt, const int *s_ustart,
                                                 const BwdArgs &a) {
    BUnit w{};
    if (MODE == kWG) {
        int g = 0;
        for (; g < a.wg_count; ++g) {
            const int mt = (a.wg_M[g] + kPairM - 1) / kPairM, nt = (a.wg_N[g] + kMaxTok - 1) / kMaxTok;
            const int ng = a.E * mt * nt;
            if (u < ng) {
                w.g = g;
                w.e = u / (mt * nt);
                const int rest = u - w.e * mt * nt;
                w.m0 = (rest / nt) * kPairM;
                w.nw0 = (rest % nt) * kMaxTok;
                break;
            }
            u -= ng;
        }
        w.kb0 = s_off[w.e] / kBlockK;
        w.kb1 = s_off[w.e + 1] / kBlockK;
        w.ntok = kMaxTok;
        return w;
    }
    constexpr int NOUT = MODE == kUV ? kPairM / 2 : kPairM;
    int lo = 0, hi = a.E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (u >= s_ustart[mid])
            lo = mid;
        else
            hi = mid - 1;
    }
    const int e = lo;
    const int local = u - s_ustart[e];
    const int ntt = s_ntt[e];
    const int tt = local % ntt;
    w.e = e;
    w.n0 = (local / ntt) * NOUT;
    const int tl = tt * s_nt[e];
    w.t0 = s_off[e] + tl;
    w.nvalid = min(s_nt[e], s_off[e + 1] - s_off[e] - tl);
    w.ntok = max(16, (w.nvalid + 15) & ~15);
    w.kb0 = 0;
    w.kb1 = MODE == kDX ? 2 * (a.ffn / kBlockK) : a.d / kBlockK;
    return w;
}

template <int MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    grouped_gemm_bwd(const __grid_constant__ BwdArgs a) {
    constexpr bool A_MN = MODE != kUV;
    constexpr bool B_MN = MODE == kWG;
    constexpr int NOUT = MODE == kUV ? kPairM / 2 : kPairM;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + kStages * kABytes;
    float *xpose = reinterpret_cast<float *>(smem + kRing);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kRing + kXpose);
    uint64_t *empty = full + kStages;
    uint64_t *acc_full = empty + kStages;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *drain = acc_empty + 2;
    uint64_t *bye = drain + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bye + 1);
    volatile int *s_abort = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *s_bye_ok = reinterpret_cast<volatile int *>(tmem_slot + 2);
    int *s_off = reinterpret_cast<int *>(tmem_slot + 4);  // [kMaxE + 1]
    int *s_ntt = s_off + kMaxE + 1;
    int *s_nt = s_ntt + kMaxE;
    int *s_ustart = s_nt + kMaxE;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();
    const bool even = rank == 0;
    const int E = a.E;

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
    pdl_wait();
    pdl_trigger();
    if (threadIdx.x <= E) s_off[threadIdx.x] = a.offsets[threadIdx.x];
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::cluster_sync_all();
    ptx::tc_fence_after_sync();
    if (threadIdx.x == 0) {
        int acc = 0;
        if (MODE == kWG) {
            for (int g = 0; g < a.wg_count; ++g)
                acc += E * ((a.wg_M[g] + kPairM - 1) / kPairM) *
                       ((a.wg_N[g] + kMaxTok - 1) / kMaxTok);
        } else {
            const int NT = ((MODE == kDX ? a.d : a.ffn) + NOUT - 1) / NOUT;
            for (int e = 0; e < E; ++e) {
                const int cnt = s_off[e + 1] - s_off[e];
                int ntt = 0, nt = 16;
                if (cnt > 0) {
                    const int t0 = (cnt + kMaxTok - 1) / kMaxTok;
                    nt = (((cnt + t0 - 1) / t0) + 15) & ~15;
                    ntt = (cnt + nt - 1) / nt;
                }
                s_ntt[e] = ntt;
                s_nt[e] = nt;
                s_ustart[e] = acc;
                acc += ntt * NT;
            }
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
            const int kbf = a.ffn / kBlockK;  // kDX: blocks of the dU W1 half
            int stage = 0;
            uint32_t ph = 0;
            int issued = 0;
            bool ok = true;
            for (int u = first; ok && u < total; u += stride) {
                const BUnit w = decode_bwd_unit<MODE>(u, s_off, s_ntt, s_nt, s_ustart, a);
                const int half = w.ntok >> 1;
                const uint32_t tx_bytes =
                    MODE == kWG ? 2u * (kABytes + kBBytes)
                                : 2u * kABytes + static_cast<uint32_t>(w.ntok) * 128u;
                const int trow = w.t0 + static_cast<int>(rank) * half;
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!ptx::mbar_wait_bounded(&empty[stage], ph ^ 1u, s_abort, a.status,
                                                kStatusProducerWait, a.wait_limit_ns)) {
                        ok = false;
                        break;
                    }
                    if (even) ptx::mbar_arrive_expect_tx(&full[stage], tx_bytes);
                    const uint32_t fb = full0 + static_cast<uint32_t>(stage) * 8u;
                    uint8_t *dA = sA + stage * kABytes;
                    uint8_t *dB = sB + stage * kBBytes;
                    const int kx = kb * kBlockK;
                    if (MODE == kUV) {
                        const int wrow = w.n0 + static_cast<int>(rank) * (kHalfM / 2);
                        ptx::tma_load_2d_pair(dA, &a.w0[w.e], kx, wrow, fb);
                        ptx::tma_load_2d_pair(dA + kBox, &a.w1[w.e], kx, wrow, fb);
                        ptx::tma_load_2d_pair(dB, &a.tok0[(half >> 3) - 1], kx, trow, fb);
                    } else if (MODE == kZ) {
                        const int c0 = w.n0 + static_cast<int>(rank) * kHalfM;
                        ptx::tma_load_2d_pair(dA, &a.w0[w.e], c0, kx, fb);
                        ptx::tma_load_2d_pair(dA + kBox, &a.w0[w.e], c0 + 64, kx, fb);
                        ptx::tma_load_2d_pair(dB, &a.tok0[(half >> 3) - 1], kx, trow, fb);
                    } else if (MODE == kDX) {
                        const int i0 = w.n0 + static_cast<int>(rank) * kHalfM;
                        const bool second = kb >= kbf;
                        const int kr = (second ? kb - kbf : kb) * kBlockK;
                        const CUtensorMap *wm = second ? &a.w1[w.e] : &a.w0[w.e];
                        ptx::tma_load_2d_pair(dA, wm, i0, kr, fb);
                        ptx::tma_load_2d_pair(dA + kBox, wm, i0 + 64, kr, fb);
                        ptx::tma_load_2d_pair(
                            dB, second ? &a.tok1[(half >> 3) - 1] : &a.tok0[(half >> 3) - 1],
                            kr, trow, fb);
                    } else {
                        const int m = w.m0 + static_cast<int>(rank) * kHalfM;
                        const int n = w.nw0 + static_cast<int>(rank) * (kMaxTok / 2);
                        ptx::tma_load_2d_pair(dA, &a.act_a[w.g], m, kx, fb);
                        ptx::tma_load_2d_pair(dA + kBox, &a.act_a[w.g], m + 64, kx, fb);
                        ptx::tma_load_2d_pair(dB, &a.act_b[w.g], n, kx, fb);
                        ptx::tma_load_2d_pair(dB + kBox, &a.act_b[w.g], n + 64, kx, fb);
                    }
                    ++issued;
                    if (++stage == kStages) {
                        stage = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (*s_abort && even) {
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
                const BUnit w = decode_bwd_unit<MODE>(u, s_off, s_ntt, s_nt, s_ustart, a);
                const uint32_t idesc = idesc_major(kPairM, w.ntok, A_MN, B_MN);
                const int acc = it & 1;
                const uint32_t aph = static_cast<uint32_t>(it >> 1) & 1u;
                if (!ptx::mbar_wait_bounded(&acc_empty[acc], aph ^ 1u, s_abort, a.status,
                                            kStatusMmaWait, a.wait_limit_ns)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc) * kAccCols;
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
                        const uint64_t ad = A_MN ? desc_mnmajor_sw128(a0 + kk * 2048)
                                                 : ptx::desc_kmajor_sw128(a0 + kk * 32);
                        const uint64_t bd = B_MN ? desc_mnmajor_sw128(b0 + kk * 2048)
                                                 : ptx::desc_kmajor_sw128(b0 + kk * 32);
                        ptx::mma_bf16_pair(d_tmem, ad, bd, idesc, (kb > w.kb0 || kk > 0) ? 1u : 0u);
                    }
                    ptx::mma_commit_pair_multicast(&empty[stage], kBothCtas);
                    if (++stage == kStages) {
                        stage = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                // (a unit with no contraction blocks issues no MMA; the commit
                // still arrives and the epilogue writes zeros)
                ptx::mma_commit_pair_multicast(&acc_full[acc], kBothCtas);
            }
            ptx::mma_commit_pair(drain);
            ptx::mbar_wait_bounded(drain, 0, nullptr, a.status, kStatusDrainWait,
                                   a.wait_limit_ns);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        // warps w, w + 4, ... read the same lane quarter (w % 4) and take
        // every (kEpiWarps / 4)-th 32-column chunk
        const int quad = warp & 3;
        const int c_first = 32 * ((warp - 2) >> 2);
        const uint32_t acc_empty0 = ptx::map_to_rank(ptx::smem_addr(&acc_empty[0]), 0);
        int it = 0;
        for (int u = first; u < total; u += stride, ++it) {
            const BUnit w = decode_bwd_unit<MODE>(u, s_off, s_ntt, s_nt, s_ustart, a);
            const int acc = it & 1;
            const uint32_t aph = static_cast<uint32_t>(it >> 1) & 1u;
            if (!ptx::mbar_wait_bounded(&acc_full[acc], aph, s_abort, a.status,
                                        kStatusEpilogueWait, a.wait_limit_ns))
                break;
            ptx::tc_fence_after_sync();
            const uint32_t tb = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                                static_cast<uint32_t>(acc) * kAccCols;
            if (MODE == kUV) {
                // lanes 0-63: U of features wrow .. +63, lanes 64-127: V of the
                // same; stored feature-major, so a thread's 32 tokens are 64
                // contiguous bytes
                const int f = w.n0 + static_cast<int>(rank) * (kHalfM / 2) + 32 * (quad & 1) + lane;
                __nv_bfloat16 *dst = (quad >= 2 ? a.V : a.U) + (size_t)f * a.rows;
                const bool f_ok = f < a.ffn;
#pragma unroll 1
                for (int j0 = c_first; j0 < w.ntok; j0 += kChunkStep) {
                    uint32_t R[32];
                    ptx::tmem_ld_32x32b_x32(tb + static_cast<uint32_t>(j0), R);
                    ptx::tmem_ld_wait();
                    if (!f_ok) continue;
                    __nv_bfloat16 *row = dst + w.t0 + j0;
                    if (j0 + 32 <= w.nvalid) {
                        uint32_t pk[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const __nv_bfloat162 b2 = __floats2bfloat162_rn(
                                __uint_as_float(R[2 * i]), __uint_as_float(R[2 * i + 1]));
                            pk[i] = *reinterpret_cast<const uint32_t *>(&b2);
                        }
                        uint4 *v4 = reinterpret_cast<uint4 *>(row);
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            v4[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (j0 + i < w.nvalid) row[i] = __float2bfloat16_rn(__uint_as_float(R[i]));
                    }
                }
            } else if (MODE == kZ) {
                const int f = w.n0 + static_cast<int>(rank) * kHalfM + 32 * quad + lane;
                const bool f_ok = f < a.ffn;
                const int fs = f_ok ? f : 0;
                const int nblk = a.ffn / 32;
                const int cb = (w.n0 + static_cast<int>(rank) * kHalfM + 32 * quad) / 32;
                const size_t ld = a.ffn;
#pragma unroll 1
                for (int j0 = c_first; j0 < w.ntok; j0 += kChunkStep) {
                    uint32_t R[32];
                    ptx::tmem_ld_32x32b_x32(tb + static_cast<uint32_t>(j0), R);
                    // lane i fetches token j0 + i's gate; the warp shares them
                    const float my_gate = j0 + lane < w.nvalid ? a.row_gate[w.t0 + j0 + lane] : 0.f;
                    ptx::tmem_ld_wait();
                    float p[32];
#pragma unroll
                    for (int hb = 0; hb < 32; hb += 16) {
                        // a half-chunk's inputs are loaded before any of its
                        // stores: 16 tokens of U and V are 32 contiguous bytes
                        // each (feature-major); a half starting below nvalid
                        // ends within the expert's 16-aligned block of rows
                        const int nv = min(16, w.nvalid - (j0 + hb));  // valid tokens in the half
                        const bool half_ok = f_ok && nv > 0;
                        const size_t fo = (size_t)fs * a.rows + w.t0 + j0 + hb;
                        const uint4 *u4 = reinterpret_cast<const uint4 *>(a.U + fo);
                        const uint4 *v4 = reinterpret_cast<const uint4 *>(a.V + fo);
                        const uint4 z4 = make_uint4(0, 0, 0, 0);
                        const uint4 uq0 = half_ok ? u4[0] : z4, uq1 = half_ok ? u4[1] : z4;
                        const uint4 vq0 = half_ok ? v4[0] : z4, vq1 = half_ok ? v4[1] : z4;
                        float ub[16], vb[16];
                        {
                            float t8[8];
                            Vec<__nv_bfloat16>::unpack(uq0, t8);
#pragma unroll
                            for (int i = 0; i < 8; ++i) ub[i] = t8[i];
                            Vec<__nv_bfloat16>::unpack(uq1, t8);
#pragma unroll
                            for (int i = 0; i < 8; ++i) ub[8 + i] = t8[i];
                            Vec<__nv_bfloat16>::unpack(vq0, t8);
#pragma unroll
                            for (int i = 0; i < 8; ++i) vb[i] = t8[i];
                            Vec<__nv_bfloat16>::unpack(vq1, t8);
#pragma unroll
                            for (int i = 0; i < 8; ++i) vb[8 + i] = t8[i];
                        }
                        const size_t ro = (size_t)(w.t0 + j0 + hb) * ld + fs;
                        __nv_bfloat16 *pdu = a.dU + ro, *pdv = a.dV + ro, *pgh = a.gH + ro;
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float z = __uint_as_float(R[hb + i]);
                            const float g = __shfl_sync(0xffffffffu, my_gate, hb + i);
                            const float uu = ub[i], vv = vb[i];
                            // logistic with the fast exponential and reciprocal:
                            // their ~1e-6 relative error vanishes next to the
                            // bf16 rounding of everything this feeds
                            const float sg = __frcp_rn(1.f + __expf(-uu));
                            const float su = uu * sg;
                            const float h = su * vv;
                            const float dh = g * z;
                            const bool ok = half_ok && i < nv;
                            p[hb + i] = ok ? h * z : 0.f;
                            if (ok) {
                                pdu[(size_t)i * ld] =
                                    __float2bfloat16_rn(dh * vv * (sg + uu * sg * (1.f - sg)));
                                pdv[(size_t)i * ld] = __float2bfloat16_rn(dh * su);
                                pgh[(size_t)i * ld] = __float2bfloat16_rn(g * h);
                            }
                        }
                    }
                    // sum over the warp's 32 features for each of the 32 tokens:
                    // halving exchanges leave lane l with token l's sum
#pragma unroll
                    for (int sft = 16; sft >= 1; sft >>= 1) {
                        const bool upper = (lane & sft) != 0;
#pragma unroll
                        for (int i = 0; i < sft; ++i) {
                            const float send = upper ? p[i] : p[i + sft];
                            const float keep = upper ? p[i + sft] : p[i];
                            p[i] = keep + __shfl_xor_sync(0xffffffffu, send, sft);
                        }
                    }
                    if (j0 + lane < w.nvalid && cb < nblk)
                        a.dgp[(size_t)(w.t0 + j0 + lane) * nblk + cb] = p[0];
                }
            } else if (MODE == kDX) {
                const int f = w.n0 + static_cast<int>(rank) * kHalfM + 32 * quad + lane;
                float *col = a.dx_rows + f;
                const bool f_ok = f < a.d;
#pragma unroll 1
                for (int j0 = c_first; j0 < w.ntok; j0 += kChunkStep) {
                    uint32_t R[32];
                    ptx::tmem_ld_32x32b_x32(tb + static_cast<uint32_t>(j0), R);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (f_ok && j0 + i < w.nvalid)
                            col[(size_t)(w.t0 + j0 + i) * a.d] = __uint_as_float(R[i]);
                }
            } else {
                // each warp holds 32 rows x 32 columns per chunk; through a
                // shared tile (rows padded to 36 floats: both phases free of
                // bank conflicts), each 16-byte store of the warp writes 4 rows
                // x 128 contiguous bytes
                const int M = a.wg_M[w.g], N = a.wg_N[w.g];
                const int mrow0 = w.m0 + static_cast<int>(rank) * kHalfM + 32 * quad;
                const bool has_k = w.kb1 > w.kb0;
                float *tile = xpose + (warp - 2) * 32 * kXpitch;
                float *out = a.wgrad[w.g][w.e];
                const int rsub = lane >> 3, c4 = (lane & 7) * 4;
#pragma unroll 1
                for (int j0 = c_first; j0 < kMaxTok; j0 += kChunkStep) {
                    uint32_t R[32];
                    ptx::tmem_ld_32x32b_x32(tb + static_cast<uint32_t>(j0), R);
                    ptx::tmem_ld_wait();
                    const int n = w.nw0 + j0;
                    if (n >= N) continue;
                    float4 *mine = reinterpret_cast<float4 *>(tile + lane * kXpitch);
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        mine[q] = has_k ? make_float4(__uint_as_float(R[4 * q]),
                                                      __uint_as_float(R[4 * q + 1]),
                                                      __uint_as_float(R[4 * q + 2]),
                                                      __uint_as_float(R[4 * q + 3]))
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
                    __syncwarp();
#pragma unroll
                    for (int r = 0; r < 8; ++r) {
                        const int row = 4 * r + rsub;
                        const float4 v = *reinterpret_cast<const float4 *>(tile + row * kXpitch + c4);
                        if (mrow0 + row < M)
                            *reinterpret_cast<float4 *>(out + (size_t)(mrow0 + row) * N + n + c4) = v;
                    }
                    __syncwarp();
                }
            }
            ptx::tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive_cluster(acc_empty0 + static_cast<uint32_t>(acc) * 8u);
        }
    }

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

std::mutex g_bwd_mutex;

template <int MODE>
int run_bwd(BwdArgs &args, int units_bound, cudaStream_t s) {
    auto kernel = grouped_gemm_bwd<MODE>;
    static bool attr_set[64];
    static int max_pairs[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
    {
        std::lock_guard<std::mutex> g(g_bwd_mutex);
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
    const int pairs = units_bound < max_pairs[dev] ? units_bound : max_pairs[dev];
    if (pairs <= 0) return MOE_OK;
    return launch_pdl(kernel, dim3(2 * pairs), kThreads, kSmem, s, args) == cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
}

int init_args(BwdArgs &args, const int *offsets, int rows, int d, int ffn, int E) {
    memset(&args, 0, sizeof args);
    args.offsets = offsets;
    args.rows = rows;
    args.d = d;
    args.ffn = ffn;
    args.E = E;
    args.wait_limit_ns = kWaitLimitNs;
    args.status = device_status_ptr();
    return args.status != nullptr ? MOE_OK : MOE_ERR_CUDA;
}

int token_maps(CUtensorMap *maps, const void *base, int rows, int K) {
    for (int i = 0; i < kTokMaps; ++i) {
        const int rc = encode_map_bf16_2d(&maps[i], base, K, rows, kBlockK, 8 * (i + 1));
        if (rc != MOE_OK) return rc;
    }
    return MOE_OK;
}

int token_units_bound(int rows, int E, int NT) { return ((rows + kMaxTok - 1) / kMaxTok + E) * NT; }

}  // namespace

int launch_bwd_uv(const void *x_rows, const int *offsets, const void *const *W1,
                  const void *const *W3, int rows, int d, int ffn, int E, void *U, void *V,
                  cudaStream_t s) {
    BwdArgs args;
    int rc = init_args(args, offsets, rows, d, ffn, E);
    if (rc == MOE_OK) rc = token_maps(args.tok0, x_rows, rows, d);
    for (int e = 0; e < E && rc == MOE_OK; ++e) {
        rc = encode_map_bf16_2d(&args.w0[e], W1[e], d, ffn, kBlockK, 64);
        if (rc == MOE_OK) rc = encode_map_bf16_2d(&args.w1[e], W3[e], d, ffn, kBlockK, 64);
    }
    if (rc != MOE_OK) return rc;
    args.U = static_cast<__nv_bfloat16 *>(U);
    args.V = static_cast<__nv_bfloat16 *>(V);
    return run_bwd<kUV>(args, token_units_bound(rows, E, (ffn + 127) / 128), s);
}

int launch_bwd_z(const void *g_rows, const int *offsets, const void *const *W2, int rows, int d,
                 int ffn, int E, const void *U, const void *V, const float *row_gate, void *dU,
                 void *dV, void *gH, float *dgp, cudaStream_t s) {
    BwdArgs args;
    int rc = init_args(args, offsets, rows, d, ffn, E);
    if (rc == MOE_OK) rc = token_maps(args.tok0, g_rows, rows, d);
    for (int e = 0; e < E && rc == MOE_OK; ++e)
        rc = encode_map_bf16_2d(&args.w0[e], W2[e], ffn, d, 64, kBlockK);
    if (rc != MOE_OK) return rc;
    args.U = const_cast<__nv_bfloat16 *>(static_cast<const __nv_bfloat16 *>(U));
    args.V = const_cast<__nv_bfloat16 *>(static_cast<const __nv_bfloat16 *>(V));
    args.row_gate = row_gate;
    args.dU = static_cast<__nv_bfloat16 *>(dU);
    args.dV = static_cast<__nv_bfloat16 *>(dV);
    args.gH = static_cast<__nv_bfloat16 *>(gH);
    args.dgp = dgp;
    return run_bwd<kZ>(args, token_units_bound(rows, E, (ffn + 255) / 256), s);
}

int launch_bwd_dx(const void *dU, const void *dV, const int *offsets, const void *const *W1,
                  const void *const *W3, int rows, int d, int ffn, int E, float *dx_rows,
                  cudaStream_t s) {
    BwdArgs args;
    int rc = init_args(args, offsets, rows, d, ffn, E);
    if (rc == MOE_OK) rc = token_maps(args.tok0, dU, rows, ffn);
    if (rc == MOE_OK) rc = token_maps(args.tok1, dV, rows, ffn);
    for (int e = 0; e < E && rc == MOE_OK; ++e) {
        rc = encode_map_bf16_2d(&args.w0[e], W1[e], d, ffn, 64, kBlockK);
        if (rc == MOE_OK) rc = encode_map_bf16_2d(&args.w1[e], W3[e], d, ffn, 64, kBlockK);
    }
    if (rc != MOE_OK) return rc;
    args.dx_rows = dx_rows;
    return run_bwd<kDX>(args, token_units_bound(rows, E, (d + 255) / 256), s);
}

int launch_bwd_wgrad(const void *x_rows, const void *g_rows, const void *dU, const void *dV,
                     const void *gH, const int *offsets, int rows, int d, int ffn, int E,
                     float *const *dW1, float *const *dW3, float *const *dW2, cudaStream_t s) {
    BwdArgs args;
    int rc = init_args(args, offsets, rows, d, ffn, E);
    // gradient 0: dW1 = dU^T X, 1: dW3 = dV^T X, 2: dW2 = G^T (g H)
    const void *A[3] = {dU, dV, g_rows};
    const void *B[3] = {x_rows, x_rows, gH};
    const int M[3] = {ffn, ffn, d}, N[3] = {d, d, ffn};
    float *const *out[3] = {dW1, dW3, dW2};
    int units = 0;
    for (int g = 0; g < 3 && rc == MOE_OK; ++g) {
        rc = encode_map_bf16_2d(&args.act_a[g], A[g], M[g], rows, 64, kBlockK);
        if (rc == MOE_OK) rc = encode_map_bf16_2d(&args.act_b[g], B[g], N[g], rows, 64, kBlockK);
        args.wg_M[g] = M[g];
        args.wg_N[g] = N[g];
        for (int e = 0; e < E; ++e) args.wgrad[g][e] = out[g][e];
        units += E * ((M[g] + kPairM - 1) / kPairM) * ((N[g] + kMaxTok - 1) / kMaxTok);
    }
    if (rc != MOE_OK) return rc;
    args.wg_count = 3;
    return run_bwd<kWG>(args, units, s);
}

size_t bwd_gemm_smem_bytes() { return kSmem; }

}  // namespace moe
