// Grouped expert GEMMs on the sm_103a tensor cores (tcgen05 + tensor memory),
// operands brought into shared memory by TMA.
//
// Each expert is a SwiGLU feed-forward network with its own weights
// ("Mixtral of Experts" (azimuth.plus), expert paragraph):
//   gate/up:  h[r][c] = silu(x_r . W1[e][c]) * (x_r . W3[e][c])   (K = d)
//   down:     y[s][r][n] = sum over split s of h[r][c] W2[e][n][c] (K = ffn)
// for every row r of expert e's contiguous block of grouped rows.
//
// Work unit = (expert, tile of up to `bm` rows, tile of output columns,
// contraction split).  A persistent grid (one CTA per SM) walks the units in
// the order expert -> column tile -> split -> row tile, so CTAs running at the
// same time share a weight tile through L2 and every weight byte of an expert
// is fetched from HBM about once.  Experts with no rows produce no units and
// their weights are never read.  The unit table is built on the device from
// `offsets`, so there is no host synchronisation.
//
// CTA = 6 warps:
//   warp 0      TMA producer (one lane): token tile + weight tile(s) per stage
//   warp 1      tensor-memory allocation; MMA issuer (one lane)
//   warps 2..5  epilogue: tensor memory -> registers -> SwiGLU / fp32 -> global
// Shared memory holds a ring of STAGES (token, weight) tile pairs; tensor
// memory holds two fp32 accumulators so the epilogue of one unit overlaps the
// MMAs of the next.
//
// The MMA is always M = 128 (one token row per tensor-memory lane).  The token
// tile copied by TMA is `bm` <= 128 rows: rows past it are never written and
// only affect accumulator lanes the epilogue never reads (row m of D depends
// only on row m of A).  For a handful of tokens (bm <= ABM < 128) a stage
// reserves only ABM token rows, so the ring holds about twice as many weight
// stages and keeps twice the bytes in flight; the MMA's reads of rows past ABM
// then land in the next slots of the ring (all token slots come first, so
// every such read stays inside the CTA's shared memory) and, again, only reach
// lanes that are never read.
//
// Every wait is bounded (see ptx::mbar_wait_bounded); on expiry the roles stop
// issuing work, drain what is in flight, free tensor memory and return, and
// the device status word records which wait expired.
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kTileM = 128;
constexpr int kMaxE = MOE_MAX_EXPERTS;
constexpr int kThreads = 192;
constexpr int kEpilogueThreads = 128;

struct TcArgs {
    CUtensorMap mapA;          // token rows [rows][K] bf16, box {64, bm}
    CUtensorMap mapB0[kMaxE];  // W1[e] (gate/up kernel) or W2[e] (down kernel): [N][K]
    CUtensorMap mapB1[kMaxE];  // W3[e] (gate/up kernel only)
    const int *offsets;        // [E + 1] expert row offsets (device)
    void *out;                 // h bf16 [rows][N]  or  y fp32 [splits][rows][N]
    int *status;               // device status word
    // gate/up split in two over the contraction (gsplit == 2; the kernel
    // takes it when it shortens the rounds of units): fp32 partial sums
    // [2][rows][2 N] (W1 half, then W3 half) and one arrival counter per
    // (expert, feature tile, token tile), zeroed before the launch
    float *gpart;
    int *gctr;
    unsigned long long wait_limit_ns;
    int E, rows, K, N, bm, kblocks, kps, splits, gsplit;
};

struct Unit {
    int e, row0, nrows, n0, ks, kb0, kb1, tile;
};

// tile: the unit's (expert, feature tile, token tile) index, the same for
// every split of it
__device__ __forceinline__ Unit decode_unit(int u, const int *s_off, const int *s_mt,
                                            const int *s_ustart, const TcArgs &a, int NOUT,
                                            int splits, int kps) {
    int e = 0;
    while (e + 1 < a.E && u >= s_ustart[e + 1]) ++e;
    const int local = u - s_ustart[e];
    const int mtn = s_mt[e];
    const int mt = local % mtn;
    const int rest = local / mtn;
    Unit w;
    w.e = e;
    w.ks = rest % splits;
    w.n0 = (rest / splits) * NOUT;
    w.row0 = s_off[e] + mt * a.bm;
    w.nrows = min(a.bm, s_off[e + 1] - w.row0);
    w.kb0 = w.ks * kps;
    w.kb1 = min(w.kb0 + kps, a.kblocks);
    w.tile = s_ustart[e] / splits + (rest / splits) * mtn + mt;
    return w;
}

template <int NB, int STAGES, int ABM>
struct SmemLayout {
    static constexpr int kABytes = ABM * 128;     // ABM token rows x 64 bf16
    static constexpr int kBBytes = NB * 128;      // NB rows x 64 bf16
    static constexpr int kRing = STAGES * (kABytes + kBBytes);
    static constexpr int kBars = (2 * STAGES + 5) * 8;
    static constexpr int kMisc = 8 + 4 * (3 * kMaxE + 5);
    static constexpr size_t kTotal = 1024 + kRing + kBars + kMisc;  // + alignment slack
    // the MMA reads 128 rows from the last token slot: past it lie weight slots
    static_assert(STAGES * kABytes + STAGES * kBBytes >= (STAGES - 1) * kABytes + kTileM * 128,
                  "MMA token reads must stay inside the ring");
    static_assert(ABM % 8 == 0 && ABM <= kTileM, "token slot of whole 8-row swizzle atoms");
};

// Named barrier 1 over the four epilogue warps; the AND form gives every
// epilogue thread the AND of their flags.
__device__ __forceinline__ void epilogue_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kEpilogueThreads) : "memory");
}

__device__ __forceinline__ bool epilogue_and(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, 1, %2, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "n"(kEpilogueThreads)
        : "memory");
    return r != 0;
}

template <int NB, int STAGES, bool SWIGLU, int ABM>
__global__ void __launch_bounds__(kThreads, 1) grouped_gemm_tc(const __grid_constant__ TcArgs a) {
    using L = SmemLayout<NB, STAGES, ABM>;
    constexpr int NOUT = SWIGLU ? NB / 2 : NB;
    // two NB-column accumulators, allocated as a power of two
    constexpr uint32_t kTmemCols = 2 * NB <= 256 ? 256 : 512;
    constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(kTileM, NB);
    static_assert(2 * NB <= 512, "two accumulators must fit tensor memory");
    static_assert(NB % 16 == 0 && NB <= 256, "MMA N for M = 128");

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + STAGES * L::kABytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::kRing);
    uint64_t *empty = full + STAGES;
    uint64_t *acc_full = empty + STAGES;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *drain = acc_empty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *s_abort = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *s_off = reinterpret_cast<int *>(tmem_slot + 2);  // [kMaxE + 1]
    int *s_mt = s_off + kMaxE + 1;                         // [kMaxE]
    int *s_ustart = s_mt + kMaxE;                          // [kMaxE + 1]
    int *s_cfg = s_ustart + kMaxE + 1;  // [0] splits, [1] 64-wide blocks a split, [2] last arrival

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = a.E;
    const int NT = (a.N + NOUT - 1) / NOUT;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&acc_full[i], 1);
            ptx::mbar_init(&acc_empty[i], kEpilogueThreads);
        }
        ptx::mbar_init(drain, 1);
        *s_abort = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(tmem_slot, kTmemCols);
        ptx::tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&a.mapA);
        ptx::prefetch_tensormap(&a.mapB0[0]);
    }
    // everything above overlaps the previous kernel's tail; the row offsets
    // and the token rows are that kernel's (or an earlier one's) output
    pdl_wait();
    pdl_trigger();
    if (threadIdx.x <= E) s_off[threadIdx.x] = a.offsets[threadIdx.x];
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    if (threadIdx.x == 0) {
        int units = 0;
        for (int e = 0; e < E; ++e) {
            const int cnt = s_off[e + 1] - s_off[e];
            const int mt = cnt > 0 ? (cnt + a.bm - 1) / a.bm : 0;
            s_mt[e] = mt;
            units += mt * NT;
        }
        int splits = a.splits, kps = a.kps;
        if (SWIGLU && a.gsplit > 1) {
            // halves of the contraction when they take fewer rounds of the
            // grid than whole units (T=1: 512 units are 4 rounds on 128 CTAs,
            // 1024 halves 7 rounds on 147 CTAs, 3.5 units' bytes each)
            const int g = (int)gridDim.x;
            const int r1 = (units + g - 1) / g, r2 = (2 * units + g - 1) / g;
            splits = r2 < 2 * r1 ? 2 : 1;
            kps = (a.kblocks + splits - 1) / splits;
        }
        int acc = 0;
        for (int e = 0; e < E; ++e) {
            s_ustart[e] = acc;
            acc += s_mt[e] * NT * splits;
        }
        s_ustart[E] = acc;
        s_cfg[0] = splits;
        s_cfg[1] = kps;
    }
    __syncthreads();
    const uint32_t tmem_base = *tmem_slot;
    const int total = s_ustart[E];
    const int splits = s_cfg[0], kps = s_cfg[1];
    // Balanced grid: the fewest rounds of units over the launched CTAs, and
    // only as many CTAs as it takes for every one to run that many (512 units
    // on 148 CTAs: 4 rounds, 128 CTAs of 4 units, rather than 68 CTAs running
    // a fourth unit alone).  An SM streams weights at about 42-50 GB/s
    // whatever the load (B300: 148 CTAs at T=16 move 6.25 TB/s, 74 CTAs
    // 3.7 TB/s), so a round run by few CTAs takes as long as a full one;
    // measured at T=1 (2 experts busy, gate/up): 148 CTAs 92.5 us, 128 CTAs
    // 86.7 us.  CTAs past the balanced count take no unit.
    const int rounds = (total + (int)gridDim.x - 1) / (int)gridDim.x;
    const int ustride = rounds > 0 ? (total + rounds - 1) / rounds : (int)gridDim.x;
    const int ufirst = (int)blockIdx.x < ustride ? (int)blockIdx.x : total;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint32_t tx_bytes = static_cast<uint32_t>(a.bm * 128 + NB * 128);
            int stage = 0;
            uint32_t ph = 0;
            int issued = 0;
            bool ok = true;
            for (int u = ufirst; ok && u < total; u += ustride) {
                const Unit w = decode_unit(u, s_off, s_mt, s_ustart, a, NOUT, splits, kps);
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!ptx::mbar_wait_bounded(&empty[stage], ph ^ 1u, s_abort, a.status,
                                                kStatusProducerWait, a.wait_limit_ns)) {
                        ok = false;
                        break;
                    }
                    uint8_t *dA = sA + stage * L::kABytes;
                    uint8_t *dB = sB + stage * L::kBBytes;
                    ptx::mbar_arrive_expect_tx(&full[stage], tx_bytes);
                    ptx::tma_load_2d(dA, &a.mapA, kb * kBlockK, w.row0, &full[stage]);
                    ptx::tma_load_2d(dB, &a.mapB0[w.e], kb * kBlockK, w.n0, &full[stage]);
                    if (SWIGLU)
                        ptx::tma_load_2d(dB + (NB / 2) * 128, &a.mapB1[w.e], kb * kBlockK, w.n0,
                                         &full[stage]);
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (*s_abort) {
                // Let copies already in flight land before the CTA exits.
                for (int i = 0; i < STAGES && i < issued; ++i) {
                    if (stage == 0) {
                        stage = STAGES - 1;
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
        if (lane == 0) {
            int stage = 0;
            uint32_t ph = 0;
            int it = 0;
            bool ok = true;
            for (int u = ufirst; ok && u < total; u += ustride, ++it) {
                const Unit w = decode_unit(u, s_off, s_mt, s_ustart, a, NOUT, splits, kps);
                const int acc = it & 1;
                const uint32_t aph = static_cast<uint32_t>(it >> 1) & 1u;
                if (!ptx::mbar_wait_bounded(&acc_empty[acc], aph ^ 1u, s_abort, a.status,
                                            kStatusMmaWait, a.wait_limit_ns)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * NB);
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!ptx::mbar_wait_bounded(&full[stage], ph, s_abort, a.status,
                                                kStatusMmaWait, a.wait_limit_ns)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after_sync();
                    const uint32_t a0 = ptx::smem_addr(sA + stage * L::kABytes);
                    const uint32_t b0 = ptx::smem_addr(sB + stage * L::kBBytes);
#pragma unroll
                    for (int kk = 0; kk < kBlockK / 16; ++kk) {
                        ptx::mma_bf16(d_tmem, ptx::desc_kmajor_sw128(a0 + kk * 32),
                                      ptx::desc_kmajor_sw128(b0 + kk * 32), kIdesc,
                                      (kb > w.kb0 || kk > 0) ? 1u : 0u);
                    }
                    ptx::mma_commit(&empty[stage]);
                    if (++stage == STAGES) {
                        stage = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                ptx::mma_commit(&acc_full[acc]);
            }
            // Every MMA issued must finish before tensor memory is released.
            ptx::mma_commit(drain);
            ptx::mbar_wait_bounded(drain, 0, nullptr, a.status, kStatusDrainWait,
                                   a.wait_limit_ns);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int quad = warp & 3;  // tensor-memory lanes 32*quad .. +31
        const int r = quad * 32 + lane;
        int it = 0;
        for (int u = ufirst; u < total; u += ustride, ++it) {
            const Unit w = decode_unit(u, s_off, s_mt, s_ustart, a, NOUT, splits, kps);
            const int acc = it & 1;
            const uint32_t aph = static_cast<uint32_t>(it >> 1) & 1u;
            // gate/up halves: partial sums out, the last half of a tile adds them
            const bool part = SWIGLU && splits > 1;
            bool ok = ptx::mbar_wait_bounded(&acc_full[acc], aph, s_abort, a.status,
                                             kStatusEpilogueWait, a.wait_limit_ns);
            // the epilogue warps meet below when splitting: they leave together
            if (part) ok = epilogue_and(ok);
            if (!ok) break;
            ptx::tc_fence_after_sync();
            const uint32_t tb =
                tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(acc * NB);
            if (quad * 32 < w.nrows) {
                const bool row_ok = r < w.nrows;
                if (part) {
                    float *prow = a.gpart +
                                  ((size_t)w.ks * a.rows + w.row0 + r) * (2 * (size_t)a.N) + w.n0;
#pragma unroll 1
                    for (int c = 0; c < NOUT; c += 32) {
                        uint32_t U[32], V[32];
                        ptx::tmem_ld_32x32b_x32(tb + c, U);
                        ptx::tmem_ld_32x32b_x32(tb + NOUT + c, V);
                        ptx::tmem_ld_wait();
                        const int nval = min(32, min(NOUT - c, a.N - (w.n0 + c)));
                        if (row_ok) {
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                if (i < nval) {
                                    prow[c + i] = __uint_as_float(U[i]);
                                    prow[a.N + c + i] = __uint_as_float(V[i]);
                                }
                        }
                    }
                } else if (SWIGLU) {
                    __nv_bfloat16 *hrow = static_cast<__nv_bfloat16 *>(a.out) +
                                          (size_t)(w.row0 + r) * a.N + w.n0;
#pragma unroll 1
                    for (int c = 0; c < NOUT; c += 32) {
                        uint32_t U[32], V[32];
                        ptx::tmem_ld_32x32b_x32(tb + c, U);
                        ptx::tmem_ld_32x32b_x32(tb + NOUT + c, V);
                        ptx::tmem_ld_wait();
                        // features of this chunk inside the tile and the
                        // matrix (NOUT = 56 leaves a chunk of 24; columns read
                        // past it are never stored)
                        const int nval = min(32, min(NOUT - c, a.N - (w.n0 + c)));
                        if (row_ok && nval > 0) {
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
                                if (8 * q < nval)
                                    dst[q] = make_uint4(packed[4 * q], packed[4 * q + 1],
                                                        packed[4 * q + 2], packed[4 * q + 3]);
                        }
                    }
                } else {
                    float *yrow = static_cast<float *>(a.out) +
                                  ((size_t)w.ks * a.rows + w.row0 + r) * a.N + w.n0;
#pragma unroll 1
                    for (int c = 0; c < NOUT; c += 32) {
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
            ptx::mbar_arrive(&acc_empty[acc]);
            if (part) {
                // the tile's last half (an arrival counter) adds the halves'
                // partial sums in split order and applies the SwiGLU
                __threadfence();
                epilogue_sync();
                if (warp == 2 && lane == 0)
                    s_cfg[2] = atomicAdd(&a.gctr[w.tile], 1) == splits - 1 ? 1 : 0;
                epilogue_sync();
                if (s_cfg[2]) {
                    __threadfence();
                    const size_t rs = 2 * (size_t)a.N, ss = (size_t)a.rows * rs;
                    for (int q = (int)threadIdx.x - 64; q < w.nrows * NOUT; q += kEpilogueThreads) {
                        const int row = q / NOUT, c = q - row * NOUT;
                        if (w.n0 + c >= a.N) continue;
                        const float *pp = a.gpart + (size_t)(w.row0 + row) * rs + w.n0 + c;
                        float uu = pp[0], vv = pp[a.N];
                        for (int s2 = 1; s2 < splits; ++s2) {
                            uu += pp[s2 * ss];
                            vv += pp[s2 * ss + a.N];
                        }
                        const float hv = uu / (1.f + expf(-uu)) * vv;
                        static_cast<__nv_bfloat16 *>(a.out)[(size_t)(w.row0 + row) * a.N + w.n0 + c] =
                            __float2bfloat16_rn(hv);
                    }
                }
            }
        }
    }

    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem_base, kTmemCols);
    }
}

std::mutex g_attr_mutex;

// Measurement override: MOE_TC_NARROW=0 keeps 128-row token slots at any bm.
bool narrow_token_slots() {
    static const bool on = [] {
        const char *v = getenv("MOE_TC_NARROW");
        return v == nullptr || atoi(v) != 0;
    }();
    return on;
}

template <int NB, int STAGES, bool SWIGLU, int ABM = kTileM>
int run_tc(TcArgs &args, int units_bound, cudaStream_t s) {
    using L = SmemLayout<NB, STAGES, ABM>;
    static_assert(L::kTotal <= 232448, "dynamic shared memory per CTA");
    if (args.bm > ABM) return MOE_ERR_ARG;
    auto kernel = grouped_gemm_tc<NB, STAGES, SWIGLU, ABM>;
    {
        // once per device, so later launches (and stream capture) only enqueue
        static bool attr_set[64];
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
        std::lock_guard<std::mutex> g(g_attr_mutex);
        if (!attr_set[dev]) {
            if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(L::kTotal)) != cudaSuccess)
                return MOE_ERR_CUDA;
            attr_set[dev] = true;
        }
    }
    int grid = units_bound < device_sm_count() ? units_bound : device_sm_count();
    // MOE_TC_GRID=n caps the persistent grid at n CTAs (measurement only)
    if (const char *g = getenv("MOE_TC_GRID"))
        if (atoi(g) > 0 && atoi(g) < grid) grid = atoi(g);
    if (grid <= 0) return MOE_OK;
    return launch_pdl(kernel, grid, kThreads, L::kTotal, s, args) == cudaSuccess ? MOE_OK
                                                                                  : MOE_ERR_CUDA;
}

int fill_common(TcArgs &args, const void *A, const int *offsets, void *out, int rows, int K,
                int N, int E, int bm) {
    args.offsets = offsets;
    args.out = out;
    args.E = E;
    args.rows = rows;
    args.K = K;
    args.N = N;
    args.bm = bm;
    args.kblocks = (K + kBlockK - 1) / kBlockK;
    args.wait_limit_ns = kWaitLimitNs;
    args.status = device_status_ptr();
    if (args.status == nullptr) return MOE_ERR_CUDA;
    return encode_map_bf16_2d(&args.mapA, A, K, rows, kBlockK, bm);
}

}  // namespace

int launch_swiglu_tc(const void *x_perm, const int *offsets, const void *const *W1,
                     const void *const *W3, int rows, int d, int ffn, int E, int bm, int wide,
                     void *h, cudaStream_t s, float *gpart, int *gctr) {
    if (rows == 0) return MOE_OK;
    TcArgs args;  // copied into the launch's parameter space at enqueue
    // few rows per expert: 112-row tiles (56 W1 + 56 W3 rows) make the Mixtral
    // shape's 8 x 256 units 13.8 waves of 148 SMs (128-row tiles: 12.1, the
    // last wave 16 SMs streaming alone)
    const int NB = wide ? 256 : 112;
    int rc = fill_common(args, x_perm, offsets, h, rows, d, ffn, E, bm);
    if (rc != MOE_OK) return rc;
    for (int e = 0; e < E; ++e) {
        if ((rc = encode_map_bf16_2d(&args.mapB0[e], W1[e], d, ffn, kBlockK, NB / 2)) != MOE_OK)
            return rc;
        if ((rc = encode_map_bf16_2d(&args.mapB1[e], W3[e], d, ffn, kBlockK, NB / 2)) != MOE_OK)
            return rc;
    }
    args.splits = 1;
    args.kps = args.kblocks;
    args.gpart = gpart;
    args.gctr = gctr;
    args.gsplit = (!wide && gpart != nullptr && gctr != nullptr) ? 2 : 1;
    const int NT = (ffn + NB / 2 - 1) / (NB / 2);
    const int units_bound = ((rows + bm - 1) / bm + E) * NT * args.gsplit;
    if (wide) return run_tc<256, 4, true>(args, units_bound, s);
    // few tokens per tile: token slots of 16/32/64 rows and more stages, about
    // 160-180 KB of ring either way (measured at 16 tokens: 6 stages of 128-row
    // slots 310.7 us, 10 or 13 stages of 16-row slots 295.5 us, 14 stages
    // 301.5 us)
    if (narrow_token_slots()) {
        if (bm <= 16) return run_tc<112, 10, true, 16>(args, units_bound, s);
        if (bm <= 32) return run_tc<112, 10, true, 32>(args, units_bound, s);
        if (bm <= 64) return run_tc<112, 8, true, 64>(args, units_bound, s);
        if (bm <= 96) return run_tc<112, 8, true, 96>(args, units_bound, s);
    }
    return run_tc<112, 6, true>(args, units_bound, s);
}

int launch_down_tc(const void *h, const int *offsets, const void *const *W2, int rows, int d,
                   int ffn, int E, int bm, int wide, int splits, int kps, float *y,
                   cudaStream_t s) {
    if (rows == 0) return MOE_OK;
    TcArgs args;
    const int NB = wide ? 256 : 128;
    int rc = fill_common(args, h, offsets, y, rows, ffn, d, E, bm);
    if (rc != MOE_OK) return rc;
    for (int e = 0; e < E; ++e)
        if ((rc = encode_map_bf16_2d(&args.mapB0[e], W2[e], ffn, d, kBlockK, NB)) != MOE_OK)
            return rc;
    args.splits = splits;
    args.kps = kps;
    args.gpart = nullptr;
    args.gctr = nullptr;
    args.gsplit = 1;
    const int NT = (d + NB - 1) / NB;
    const int units_bound = ((rows + bm - 1) / bm + E) * NT * splits;
    if (wide) return run_tc<256, 4, false>(args, units_bound, s);
    // (measured at 16 tokens: 6, 8, 10, 12 stages of 16-row slots 153.2, 149.4,
    // 147.5, 155.7 us; 6 stages of 128-row slots 153.0 us)
    if (narrow_token_slots()) {
        if (bm <= 16) return run_tc<128, 10, false, 16>(args, units_bound, s);
        if (bm <= 32) return run_tc<128, 9, false, 32>(args, units_bound, s);
        if (bm <= 64) return run_tc<128, 7, false, 64>(args, units_bound, s);
        if (bm <= 96) return run_tc<128, 8, false, 96>(args, units_bound, s);
    }
    return run_tc<128, 6, false>(args, units_bound, s);
}

}  // namespace moe
