// Grouped expert GEMMs on CTA pairs with the tokens as the MMA's N side.
//
// Same operation as gemm_tc.cu (gate/up with the SwiGLU epilogue, or the down
// projection), organised for tensor-core efficiency when experts hold many
// rows:
//   - a cluster of two CTAs on neighbouring SMs issues tcgen05 .cta_group::2
//     MMAs of M = 256 weight rows (128 in each CTA's shared memory) by
//     N = up to 256 token rows (half in each CTA);
//   - an expert's rows are cut into ceil(cnt / 256) token tiles of equal size
//     rounded up to 16, the MMA's N granularity, so at most 15 padded rows per
//     tile reach the tensor cores (a 128- or 256-row M tile pads up to 127 or
//     255 at each expert's tail);
//   - gate/up: each CTA's 128 weight rows are 64 rows of W1 and the same 64
//     rows of W3 (two TMA boxes), so the gate of feature f sits in
//     accumulator lane f and its up value in lane 64 + f, in another warp's
//     quarter; the two warps swap half of each 32-token chunk through shared
//     memory and each finishes silu(u) * v for 16 of the tokens;
//   - down: each CTA holds 128 of the pair's 256 output features.
// The accumulator is feature-major (lane = feature, column = token), so the
// epilogue writes, per token, 32 consecutive features from one warp.
//
// Roles: warp 0 issues TMA copies, warp 1 the MMAs (even CTA), warps 2-9 are
// the epilogue: two warps per tensor-memory lane quarter taking alternate
// 32-token chunks.
//
// Barriers (same offsets in both CTAs):
//   full[s]      even CTA only: one arrival with the stage's byte count from
//                the even CTA's producer; both CTAs' TMA copies complete
//                bytes on it;
//   empty[s]     both CTAs: the even CTA's MMA commit multicasts to both;
//   acc_full[a]  both CTAs: MMA commit multicast, read by each epilogue;
//   acc_empty[a] even CTA only: one arrival per epilogue warp of both CTAs (16);
//   drain, bye   teardown: the MMA drain, and a pair handshake so neither CTA
//                leaves while the other may still touch its shared memory.
// Every wait is bounded as in gemm_tc.cu.
#include <stdlib.h>

#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kPairM = 256;        // weight rows per pair tile
constexpr int kHalfM = 128;        // weight rows per CTA
constexpr int kMaxTok = 256;       // token rows per tile (MMA N)
constexpr int kTokMaps = kMaxTok / 16;  // token tensor maps, box heights 8, 16, ..., 128
constexpr int kGate = kHalfM / 2;  // gate/up: W1 rows, then the same rows of W3, per CTA
constexpr int kMaxE = MOE_MAX_EXPERTS;
constexpr int kEpiWarps = 8;  // two per tensor-memory lane quarter
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kABytes = kHalfM * 128;       // weights, 64-wide contraction slice
constexpr int kBBytes = (kMaxTok / 2) * 128;  // tokens, this CTA's half
// gate/up exchange (two-box layout): [warp pair 4][chunk parity 2][direction 2]
// [16 tokens][32 lanes] fp32
constexpr int kXchPairs = kEpiWarps / 2;
constexpr int kXchFloats = 16 * 32;
constexpr int kXch = kXchPairs * 2 * 2 * kXchFloats * 4;
constexpr int kMisc = 16 + 4 * (4 * kMaxE + 2);

// Shared memory of one instantiation.  Gate/up with the two-box weight layout
// needs the 32 KB exchange and keeps six ring stages; the interleaved layout
// (IL) and the down projection need no exchange and take a seventh stage.
template <bool SWIGLU, bool IL>
struct PairCfg {
    static constexpr bool kXchOn = SWIGLU && !IL;
    static constexpr int kStages = kXchOn ? 6 : 7;
    static constexpr int kRing = kStages * (kABytes + kBBytes);
    static constexpr int kXchBytes = kXchOn ? kXch : 0;
    static constexpr int kBars = (2 * kStages + 6 + (kXchOn ? kXchPairs : 0)) * 8;
    static constexpr size_t kSmem = 1024 + kRing + kXchBytes + kBars + kMisc;
    static_assert(kSmem <= 232448, "dynamic shared memory of one CTA");
};
constexpr uint32_t kAccCols = kMaxTok;
constexpr uint32_t kTmemCols = 2 * kAccCols;
constexpr int kAccEmptyArrivals = 2 * kEpiWarps;  // lane 0 of each epilogue warp, both CTAs
constexpr uint16_t kBothCtas = 0x3;

struct PairArgs {
    CUtensorMap mapTok[kTokMaps];  // token rows [rows][K] bf16; map i has box {64, 8 (i + 1)}
    CUtensorMap mapW0[kMaxE];      // W1[e] (gate/up, box {64, 64}) or W2[e] (down, box {64, 128})
    CUtensorMap mapW1[kMaxE];      // W3[e] (gate/up only, box {64, 64})
    const int *offsets;            // [E + 1]
    void *out;                     // h bf16 [rows][N], y fp32 [splits][rows][N],
                                   // or (combine) acc fp32 [T][N]
    const int *perm;               // combine: row -> token * k + slot
    const float *gates;            // combine: [T][k]
    int *status;
    unsigned long long wait_limit_ns;
    int E, rows, K, N, kblocks, kps, splits;
    int k;        // combine: experts per token
    int combine;  // down only: add gate x output into acc[token] (one split)
    // interleaved gate/up: mapW0[e] is the 4-D map of W1[e] and W3[e] (box
    // {64, 16, 2, 4}); bit e set when W3[e]'s rows come first in each group
    unsigned long long swap_mask;
    int balance;  // balanced grid (see the kernel)
};

struct PairUnit {
    int e;       // expert
    int t0;      // first token row of the tile (row of x_perm / h)
    int nvalid;  // token rows in the tile
    int ntok;    // MMA N: nvalid rounded up to 16
    int n0;      // first output feature of the pair's tile
    int ks, kb0, kb1;  // contraction split and its 64-wide blocks
};

// Units are ordered expert -> feature tile -> split -> token tile, so the
// pairs running together share one weight tile through L2.  (Feature tile
// first, spreading the pairs running together over the experts, measured
// 1-10% slower at T = 512 .. 4096.)
__device__ __forceinline__ PairUnit decode_pair_unit(int u, const int *s_off, const int *s_ntt,
                                                     const int *s_nt, const int *s_ustart,
                                                     const PairArgs &a, int NOUT) {
    int lo = 0, hi = a.E - 1;
    while (lo < hi) {  // last expert whose first unit is <= u (experts with no units share it)
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
    const int rest = local / ntt;
    PairUnit w;
    w.e = e;
    w.ks = rest % a.splits;
    w.n0 = (rest / a.splits) * NOUT;
    const int tl = tt * s_nt[e];
    w.t0 = s_off[e] + tl;
    w.nvalid = min(s_nt[e], s_off[e + 1] - s_off[e] - tl);
    w.ntok = max(16, (w.nvalid + 15) & ~15);
    w.kb0 = w.ks * a.kps;
    w.kb1 = min(w.kb0 + a.kps, a.kblocks);
    return w;
}

template <bool SWIGLU, bool IL>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    grouped_gemm_pair(const __grid_constant__ PairArgs a) {
    constexpr int NOUT = SWIGLU ? kPairM / 2 : kPairM;  // output features per pair tile
    using C = PairCfg<SWIGLU, IL>;
    constexpr int kStages = C::kStages;
    constexpr int kRing = C::kRing;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + kStages * kABytes;
    float *xch = reinterpret_cast<float *>(smem + kRing);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kRing + C::kXchBytes);
    uint64_t *empty = full + kStages;
    uint64_t *acc_full = empty + kStages;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *drain = acc_empty + 2;
    uint64_t *bye = drain + 1;
    uint64_t *xbar = bye + 1;  // [kXchPairs] gate/up exchange (two-box layout)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(xbar + (C::kXchOn ? kXchPairs : 0));
    volatile int *s_abort = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *s_bye_ok = reinterpret_cast<volatile int *>(tmem_slot + 2);
    int *s_off = reinterpret_cast<int *>(tmem_slot + 4);  // [kMaxE + 1]
    int *s_ntt = s_off + kMaxE + 1;                        // [kMaxE] token tiles
    int *s_nt = s_ntt + kMaxE;                             // [kMaxE] rows per token tile
    int *s_ustart = s_nt + kMaxE;                          // [kMaxE + 1]

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
        if (C::kXchOn)
            for (int i = 0; i < kXchPairs; ++i) ptx::mbar_init(&xbar[i], 2);
        *s_abort = 0;
        *s_bye_ok = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc_pair(tmem_slot, kTmemCols);
        ptx::tmem_relinquish_pair();
    }
    if (warp == 0 && lane == 0) {
        for (int i = 0; i < kTokMaps; ++i) ptx::prefetch_tensormap(&a.mapTok[i]);
    }
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
            int ntt = 0, nt = 16;
            if (cnt > 0) {
                const int t0 = (cnt + kMaxTok - 1) / kMaxTok;
                nt = (((cnt + t0 - 1) / t0) + 15) & ~15;  // <= kMaxTok
                ntt = (cnt + nt - 1) / nt;
            }
            s_ntt[e] = ntt;
            s_nt[e] = nt;
            s_ustart[e] = acc;
            acc += ntt * NT * a.splits;
        }
        s_ustart[E] = acc;
    }
    __syncthreads();
    const uint32_t tmem_base = *tmem_slot;
    const int total = s_ustart[E];
    // Balanced grid (as in gemm_tc.cu): the fewest rounds of units over the
    // launched pairs, and only as many pairs as it takes for every one to
    // run that many; pairs past that count take no unit.  MOE_PAIR_BALANCE
    // (a kernel argument) turns it off for measurement.
    const int npairs = static_cast<int>(ptx::cluster_count_x());
    const int rounds = (total + npairs - 1) / npairs;
    const int stride = (a.balance && rounds > 0) ? (total + rounds - 1) / rounds : npairs;
    const int cid = static_cast<int>(ptx::cluster_id_x());
    const int first = cid < stride ? cid : total;

    if (warp == 0) {
        // ------------------------------------------------------------ producers
        if (lane == 0) {
            const uint32_t full0 = ptx::map_to_rank(ptx::smem_addr(&full[0]), 0);
            int stage = 0;
            uint32_t ph = 0;
            int issued = 0;
            bool ok = true;
            for (int u = first; ok && u < total; u += stride) {
                const PairUnit w = decode_pair_unit(u, s_off, s_ntt, s_nt, s_ustart, a, NOUT);
                const int half = w.ntok >> 1;  // token rows this CTA supplies
                const CUtensorMap *mt = &a.mapTok[(half >> 3) - 1];
                const uint32_t tx_bytes = 2u * kABytes + static_cast<uint32_t>(w.ntok) * 128u;
                const int trow = w.t0 + static_cast<int>(rank) * half;
                const int wrow = w.n0 + static_cast<int>(rank) * (SWIGLU ? kGate : kHalfM);
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!ptx::mbar_wait_bounded(&empty[stage], ph ^ 1u, s_abort, a.status,
                                                kStatusProducerWait, a.wait_limit_ns)) {
                        ok = false;
                        break;
                    }
                    if (even) ptx::mbar_arrive_expect_tx(&full[stage], tx_bytes);
                    const uint32_t fb = full0 + static_cast<uint32_t>(stage) * 8u;
                    uint8_t *dA = sA + stage * kABytes;
                    const int kx = kb * kBlockK;
                    if (IL) {
                        // 128 rows: four groups of 16 gate and the same 16 up rows
                        ptx::tma_load_4d_pair(dA, &a.mapW0[w.e], kx, 0, 0, wrow / 16, fb);
                    } else {
                        ptx::tma_load_2d_pair(dA, &a.mapW0[w.e], kx, wrow, fb);
                        if (SWIGLU)
                            ptx::tma_load_2d_pair(dA + kGate * 128, &a.mapW1[w.e], kx, wrow, fb);
                    }
                    ptx::tma_load_2d_pair(sB + stage * kBBytes, mt, kx, trow, fb);
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
                const PairUnit w = decode_pair_unit(u, s_off, s_ntt, s_nt, s_ustart, a, NOUT);
                const uint32_t idesc = ptx::idesc_bf16_f32(kPairM, w.ntok);
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
                        ptx::mma_bf16_pair(d_tmem, ptx::desc_kmajor_sw128(a0 + kk * 32),
                                           ptx::desc_kmajor_sw128(b0 + kk * 32), idesc,
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
        // warps w and w + 4 read the same lane quarter and take alternate
        // 32-token chunks
        const int cset = (warp - 2) >> 2;
        const uint32_t acc_empty0 = ptx::map_to_rank(ptx::smem_addr(&acc_empty[0]), 0);
        // gate/up: quarters 0 and 1 hold the gate values of features 0-31 and
        // 32-63, quarters 2 and 3 the up values of the same features
        const int pairq = (quad & 1) + 2 * cset;
        const bool is_up = quad >= 2;
        float *xb = xch + pairq * (2 * 2 * kXchFloats);
        uint32_t xk = 0;  // exchanges done by this warp pair
        bool ok = true;
        int it = 0;
        for (int u = first; ok && u < total; u += stride, ++it) {
            const PairUnit w = decode_pair_unit(u, s_off, s_ntt, s_nt, s_ustart, a, NOUT);
            const int acc = it & 1;
            const uint32_t aph = static_cast<uint32_t>(it >> 1) & 1u;
            if (!ptx::mbar_wait_bounded(&acc_full[acc], aph, s_abort, a.status,
                                        kStatusEpilogueWait, a.wait_limit_ns))
                break;
            ptx::tc_fence_after_sync();
            const uint32_t tb = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                                static_cast<uint32_t>(acc) * kAccCols;
            if (IL) {
                // interleaved rows: lanes 0-15 of this quarter hold one
                // matrix's values of features 16 quad .. +15, lanes 16-31 the
                // other's of the same features; lane pairs (l, l + 16) swap
                // half of each 32-token chunk by shuffle and each finishes
                // silu(u) * v for 16 tokens
                const bool upper = lane >= 16;
                const bool is_gate = upper == (((a.swap_mask >> w.e) & 1ull) != 0);
                const int f = w.n0 + static_cast<int>(rank) * kGate + quad * 16 + (lane & 15);
                __nv_bfloat16 *hcol = static_cast<__nv_bfloat16 *>(a.out) + f;
                const bool f_ok = f < a.N;
#pragma unroll 1
                for (int j0 = 32 * cset; j0 < w.ntok; j0 += 64) {
                    uint32_t V[32];
                    ptx::tmem_ld_32x32b_x32(tb + static_cast<uint32_t>(j0), V);
                    ptx::tmem_ld_wait();
                    // the gate lane keeps tokens 0-15 of the chunk, the up lane 16-31
                    const int jb = j0 + (is_gate ? 0 : 16);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float send = __uint_as_float(is_gate ? V[16 + i] : V[i]);
                        const float other = __shfl_xor_sync(0xffffffffu, send, 16);
                        const float g = is_gate ? __uint_as_float(V[i]) : other;
                        const float v = is_gate ? other : __uint_as_float(V[16 + i]);
                        const int j = jb + i;
                        if (f_ok && j < w.nvalid)
                            hcol[(size_t)(w.t0 + j) * a.N] =
                                __float2bfloat16_rn(g / (1.f + expf(-g)) * v);
                    }
                }
            } else if (SWIGLU) {
                // the gate warp finishes each chunk's first 16 tokens, the up
                // warp the last 16; each sends the other the values it needs
                const int f = w.n0 + static_cast<int>(rank) * kGate + (quad & 1) * 32 + lane;
                __nv_bfloat16 *hcol = static_cast<__nv_bfloat16 *>(a.out) + f;
                const bool f_ok = f < a.N;
#pragma unroll 1
                for (int j0 = 32 * cset; j0 < w.ntok; j0 += 64) {
                    uint32_t V[32];
                    ptx::tmem_ld_32x32b_x32(tb + static_cast<uint32_t>(j0), V);
                    ptx::tmem_ld_wait();
                    float *buf = xb + (xk & 1u) * (2 * kXchFloats);
                    float *send = buf + (is_up ? kXchFloats : 0);
                    const float *recv = buf + (is_up ? 0 : kXchFloats);
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        send[i * 32 + lane] = __uint_as_float(is_up ? V[i] : V[16 + i]);
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(&xbar[pairq]);
                    if (!ptx::mbar_wait_bounded(&xbar[pairq], xk & 1u, s_abort, a.status,
                                                kStatusEpilogueWait, a.wait_limit_ns)) {
                        ok = false;
                        break;
                    }
                    ++xk;
                    const int jb = j0 + (is_up ? 16 : 0);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float other = recv[i * 32 + lane];
                        const float g = is_up ? other : __uint_as_float(V[i]);
                        const float v = is_up ? __uint_as_float(V[16 + i]) : other;
                        const int j = jb + i;
                        if (f_ok && j < w.nvalid)
                            hcol[(size_t)(w.t0 + j) * a.N] =
                                __float2bfloat16_rn(g / (1.f + expf(-g)) * v);
                    }
                }
                if (!ok) break;
            } else if (a.combine) {
                // the combine: each of the chunk's rows adds gate x output into
                // its token's accumulator row (lane i fetches row i's token and
                // gate, shared across the warp)
                const int f = w.n0 + static_cast<int>(rank) * kHalfM + quad * 32 + lane;
                float *acol = static_cast<float *>(a.out) + f;
                const bool f_ok = f < a.N;
#pragma unroll 1
                for (int j0 = 32 * cset; j0 < w.ntok; j0 += 64) {
                    uint32_t Y[32];
                    ptx::tmem_ld_32x32b_x32(tb + static_cast<uint32_t>(j0), Y);
                    int my_tok = 0;
                    float my_gate = 0.f;
                    if (j0 + lane < w.nvalid) {
                        const int p = a.perm[w.t0 + j0 + lane];
                        my_tok = a.k == 2 ? (p >> 1) : p / a.k;
                        my_gate = a.gates[p];
                    }
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int tok = __shfl_sync(0xffffffffu, my_tok, i);
                        const float g = __shfl_sync(0xffffffffu, my_gate, i);
                        if (f_ok && j0 + i < w.nvalid)
                            atomicAdd(acol + (size_t)tok * a.N, g * __uint_as_float(Y[i]));
                    }
                }
            } else {
                const int f = w.n0 + static_cast<int>(rank) * kHalfM + quad * 32 + lane;
                float *ycol = static_cast<float *>(a.out) + (size_t)w.ks * a.rows * a.N + f;
                const bool f_ok = f < a.N;
#pragma unroll 1
                for (int j0 = 32 * cset; j0 < w.ntok; j0 += 64) {
                    uint32_t Y[32];
                    ptx::tmem_ld_32x32b_x32(tb + static_cast<uint32_t>(j0), Y);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int j = j0 + i;
                        if (f_ok && j < w.nvalid)
                            ycol[(size_t)(w.t0 + j) * a.N] = __uint_as_float(Y[i]);
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

template <bool SWIGLU, bool IL = false>
int run_pair(PairArgs &args, int units_bound, cudaStream_t s) {
    auto kernel = grouped_gemm_pair<SWIGLU, IL>;
    constexpr size_t kSmem = PairCfg<SWIGLU, IL>::kSmem;
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

// Token maps (one per tile height), shapes and the status word.
int fill_pair(PairArgs &args, const void *tokens, const int *offsets, void *out, int rows, int K,
              int N, int E) {
    args.offsets = offsets;
    args.out = out;
    args.perm = nullptr;
    args.gates = nullptr;
    args.k = 1;
    args.combine = 0;
    args.swap_mask = 0;
    // MOE_PAIR_BALANCE=0 turns the balanced grid off (measurement only)
    args.balance = 1;
    if (const char *b = getenv("MOE_PAIR_BALANCE")) args.balance = atoi(b) != 0;
    args.E = E;
    args.rows = rows;
    args.K = K;
    args.N = N;
    args.kblocks = (K + kBlockK - 1) / kBlockK;
    args.wait_limit_ns = kWaitLimitNs;
    args.status = device_status_ptr();
    if (args.status == nullptr) return MOE_ERR_CUDA;
    for (int i = 0; i < kTokMaps; ++i) {
        const int rc = encode_map_bf16_2d(&args.mapTok[i], tokens, K, rows, kBlockK, 8 * (i + 1));
        if (rc != MOE_OK) return rc;
    }
    return MOE_OK;
}

// Upper bound on the token tiles of all experts together.
int token_tiles_bound(int rows, int E) { return (rows + kMaxTok - 1) / kMaxTok + E; }

}  // namespace

size_t pair_gemm_smem_bytes() {
    return PairCfg<true, false>::kSmem > PairCfg<false, false>::kSmem
               ? PairCfg<true, false>::kSmem
               : PairCfg<false, false>::kSmem;
}

int launch_swiglu_pair(const void *x_perm, const int *offsets, const void *const *W1,
                       const void *const *W3, int rows, int d, int ffn, int E, void *h,
                       cudaStream_t s) {
    if (rows == 0) return MOE_OK;
    PairArgs args;
    int rc = fill_pair(args, x_perm, offsets, h, rows, d, ffn, E);
    if (rc != MOE_OK) return rc;
    args.splits = 1;
    args.kps = args.kblocks;
    const int NT = (ffn + kPairM / 2 - 1) / (kPairM / 2);
    // W1[e] and W3[e] interleaved by one 4-D map per expert (seven stages, no
    // exchange buffer), unless the driver refuses that layout for some
    // expert; MOE_PAIR_IL=0 forces the two-box layout (measurement only)
    bool il = true;
    if (const char *v = getenv("MOE_PAIR_IL")) il = atoi(v) != 0;
    for (int e = 0; il && e < E; ++e) {
        int sw = 0;
        rc = encode_map_gate_up(&args.mapW0[e], W1[e], W3[e], d, ffn, &sw);
        if (rc == MOE_ERR_UNSUPPORTED) il = false;
        else if (rc != MOE_OK) return rc;
        if (sw) args.swap_mask |= 1ull << e;
    }
    if (il) return run_pair<true, true>(args, token_tiles_bound(rows, E) * NT, s);
    args.swap_mask = 0;
    for (int e = 0; e < E; ++e) {
        if ((rc = encode_map_bf16_2d(&args.mapW0[e], W1[e], d, ffn, kBlockK, kGate)) != MOE_OK)
            return rc;
        if ((rc = encode_map_bf16_2d(&args.mapW1[e], W3[e], d, ffn, kBlockK, kGate)) != MOE_OK)
            return rc;
    }
    return run_pair<true, false>(args, token_tiles_bound(rows, E) * NT, s);
}

int launch_down_pair(const void *h, const int *offsets, const void *const *W2, int rows, int d,
                     int ffn, int E, int splits, int kps, float *y, cudaStream_t s) {
    if (rows == 0) return MOE_OK;
    PairArgs args;
    int rc = fill_pair(args, h, offsets, y, rows, ffn, d, E);
    if (rc != MOE_OK) return rc;
    for (int e = 0; e < E; ++e)
        if ((rc = encode_map_bf16_2d(&args.mapW0[e], W2[e], ffn, d, kBlockK, kHalfM)) != MOE_OK)
            return rc;
    args.splits = splits;
    args.kps = kps;
    const int NT = (d + kPairM - 1) / kPairM;
    return run_pair<false>(args, token_tiles_bound(rows, E) * NT * splits, s);
}

int launch_down_pair_combine(const void *h, const int *offsets, const void *const *W2, int rows,
                             int d, int ffn, int E, const int *perm, const float *gates, int k,
                             float *acc, cudaStream_t s) {
    if (rows == 0) return MOE_OK;
    if (k < 1 || k > 2 || perm == nullptr || gates == nullptr) return MOE_ERR_ARG;
    PairArgs args;
    int rc = fill_pair(args, h, offsets, acc, rows, ffn, d, E);
    if (rc != MOE_OK) return rc;
    for (int e = 0; e < E; ++e)
        if ((rc = encode_map_bf16_2d(&args.mapW0[e], W2[e], ffn, d, kBlockK, kHalfM)) != MOE_OK)
            return rc;
    args.splits = 1;
    args.kps = args.kblocks;
    args.perm = perm;
    args.gates = gates;
    args.k = k;
    args.combine = 1;
    const int NT = (d + kPairM - 1) / kPairM;
    return run_pair<false>(args, token_tiles_bound(rows, E) * NT, s);
}

}  // namespace moe
