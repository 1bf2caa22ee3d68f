// C ABI of libmoe.so: argument checks, the per-call plan (tiles, splits,
// workspace layout) and the sequence of kernel launches.  See include/moe.h.
#include <cudaTypedefs.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>
#include <string>
#include <unordered_map>

#include "internal.h"

namespace moe {

// Status word written by kernels whose bounded waits expire.
__device__ int g_device_status = 0;

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Host-side fault injection for tests of the error paths: MOE_FAULT_INJECT
// set to "arg", "workspace" or "cuda" makes the next checked entry point fail
// with that error before anything is enqueued.
int injected_fault() {
    const char *f = getenv("MOE_FAULT_INJECT");
    if (f == nullptr || f[0] == '\0') return MOE_OK;
    if (strcmp(f, "arg") == 0) return MOE_ERR_ARG;
    if (strcmp(f, "workspace") == 0) return MOE_ERR_WORKSPACE;
    if (strcmp(f, "cuda") == 0) return MOE_ERR_CUDA;
    return MOE_OK;
}

int check_dims(int T, int d, int ffn, int E, int k, int dt) {
    if (T < 0 || d <= 0 || ffn <= 0 || E <= 0 || k <= 0 || k > E) return MOE_ERR_ARG;
    if (dt != MOE_F32 && dt != MOE_BF16) return MOE_ERR_ARG;
    if (E > MOE_MAX_EXPERTS || k > MOE_MAX_TOPK) return MOE_ERR_UNSUPPORTED;
    if (dt == MOE_BF16 && (d % 64 != 0 || ffn % 64 != 0)) return MOE_ERR_UNSUPPORTED;
    if (dt == MOE_F32 && (d % 4 != 0 || ffn % 4 != 0)) return MOE_ERR_UNSUPPORTED;
    // index arithmetic is 32-bit for rows and 64-bit for element offsets
    if ((long long)T * k > (1ll << 30)) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

int check_weights(const void *const *W, int E) {
    if (W == nullptr) return MOE_ERR_ARG;
    for (int e = 0; e < E; ++e) {
        if (W[e] == nullptr) return MOE_ERR_ARG;
        if (!aligned16(W[e])) return MOE_ERR_UNSUPPORTED;
    }
    return MOE_OK;
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

std::mutex g_dev_mutex;
int g_sm_count[64];
int *g_status_ptr[64];

int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
    return dev;
}

}  // namespace

int elem_size(int dt) { return dt == MOE_BF16 ? 2 : 4; }

// Measured on B300 (bench.py, same box): decode unchanged, prefill about 2.5%
// slower with the overlap, so it is off unless MOE_PDL=1.
bool pdl_enabled() {
    static const bool on = [] {
        const char *v = getenv("MOE_PDL");
        return v != nullptr && v[0] == '1';
    }();
    return on;
}

int device_sm_count() {
    const int dev = current_device();
    if (dev < 0) return kPlanSms;
    std::lock_guard<std::mutex> g(g_dev_mutex);
    if (g_sm_count[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            n <= 0)
            n = kPlanSms;
        g_sm_count[dev] = n;
    }
    return g_sm_count[dev];
}

int *device_status_ptr() {
    const int dev = current_device();
    if (dev < 0) return nullptr;
    std::lock_guard<std::mutex> g(g_dev_mutex);
    if (g_status_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<int *>(p);
    }
    return g_status_ptr[dev];
}

namespace {

// Encoded tensor maps, keyed by everything that goes into one.  A map depends
// only on these values, so a cached entry is always valid; the cache is
// emptied when it grows past kMapCacheMax entries.
struct MapKey {
    const void *base;
    unsigned long long inner, outer;
    unsigned int box_inner, box_outer;
    bool operator==(const MapKey &o) const {
        return base == o.base && inner == o.inner && outer == o.outer &&
               box_inner == o.box_inner && box_outer == o.box_outer;
    }
};

struct MapKeyHash {
    size_t operator()(const MapKey &k) const {
        size_t h = std::hash<const void *>()(k.base);
        h ^= std::hash<unsigned long long>()(k.inner * 1000003ull + k.outer) + 0x9e3779b97f4a7c15ull +
             (h << 6) + (h >> 2);
        h ^= std::hash<unsigned long long>()(((unsigned long long)k.box_inner << 32) | k.box_outer) +
             0x9e3779b97f4a7c15ull + (h << 6) + (h >> 2);
        return h;
    }
};

constexpr size_t kMapCacheMax = 8192;
std::mutex g_map_mutex;
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_map_cache;

int encode_uncached(CUtensorMap *map, const void *base, unsigned long long inner,
                    unsigned long long outer, unsigned int box_inner, unsigned int box_outer);

}  // namespace

int encode_map_bf16_2d(CUtensorMap *map, const void *base, unsigned long long inner,
                       unsigned long long outer, unsigned int box_inner, unsigned int box_outer) {
    const MapKey key{base, inner, outer, box_inner, box_outer};
    {
        std::lock_guard<std::mutex> g(g_map_mutex);
        auto it = g_map_cache.find(key);
        if (it != g_map_cache.end()) {
            *map = it->second;
            return MOE_OK;
        }
    }
    const int rc = encode_uncached(map, base, inner, outer, box_inner, box_outer);
    if (rc == MOE_OK) {
        std::lock_guard<std::mutex> g(g_map_mutex);
        if (g_map_cache.size() >= kMapCacheMax) g_map_cache.clear();
        g_map_cache.emplace(key, *map);
    }
    return rc;
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return encode;
}

struct GateUpKey {
    const void *w1, *w3;
    int d, ffn;
    bool operator==(const GateUpKey &o) const {
        return w1 == o.w1 && w3 == o.w3 && d == o.d && ffn == o.ffn;
    }
};

struct GateUpKeyHash {
    size_t operator()(const GateUpKey &k) const {
        size_t h = std::hash<const void *>()(k.w1);
        h ^= std::hash<const void *>()(k.w3) + 0x9e3779b97f4a7c15ull + (h << 6) + (h >> 2);
        h ^= std::hash<long long>()(((long long)k.d << 32) | (unsigned)k.ffn) +
             0x9e3779b97f4a7c15ull + (h << 6) + (h >> 2);
        return h;
    }
};

struct GateUpMap {
    CUtensorMap map;
    int swapped;
};

std::unordered_map<GateUpKey, GateUpMap, GateUpKeyHash> g_gate_up_cache;

int encode_uncached(CUtensorMap *map, const void *base, unsigned long long inner,
                    unsigned long long outer, unsigned int box_inner, unsigned int box_outer) {
    const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (encode == nullptr) return MOE_ERR_CUDA;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {inner * 2};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base),
                              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace

// W1[e] and W3[e] ([ffn][d] each) as one 4-D tensor: dims (d, 16 rows, 2
// matrices, ffn / 16 row groups), strides (2 d bytes, the distance from the
// lower of the two matrices to the higher, 32 d bytes).  A box {64, 16, 2, 4}
// lands in shared memory as four groups of [16 rows of one matrix, the same
// 16 rows of the other]: 128 rows whose gate and up values of a feature sit
// 16 rows apart.  *swapped = 1 when W3[e] lies below W1[e] (the box then puts
// W3's rows first).  Returns MOE_ERR_UNSUPPORTED when the driver refuses the
// layout (the caller falls back to two separate boxes).
int encode_map_gate_up(CUtensorMap *map, const void *W1e, const void *W3e, int d, int ffn,
                       int *swapped) {
    const GateUpKey key{W1e, W3e, d, ffn};
    {
        std::lock_guard<std::mutex> g(g_map_mutex);
        auto it = g_gate_up_cache.find(key);
        if (it != g_gate_up_cache.end()) {
            *map = it->second.map;
            *swapped = it->second.swapped;
            return MOE_OK;
        }
    }
    const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (encode == nullptr) return MOE_ERR_CUDA;
    if (ffn % 64 != 0 || W1e == W3e) return MOE_ERR_UNSUPPORTED;
    const uintptr_t a = reinterpret_cast<uintptr_t>(W1e), b = reinterpret_cast<uintptr_t>(W3e);
    const int sw = b < a ? 1 : 0;
    const uintptr_t lo = sw ? b : a, hi = sw ? a : b;
    const unsigned long long gap = static_cast<unsigned long long>(hi - lo);
    if (gap % 16 != 0 || gap >= (1ull << 40)) return MOE_ERR_UNSUPPORTED;
    const cuuint64_t dims[4] = {(cuuint64_t)d, 16, 2, (cuuint64_t)(ffn / 16)};
    const cuuint64_t strides[3] = {(cuuint64_t)d * 2, gap, (cuuint64_t)d * 2 * 16};
    const cuuint32_t box[4] = {64, 16, 2, 4};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUtensorMap m;
    const CUresult r = encode(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                              reinterpret_cast<void *>(lo), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return MOE_ERR_UNSUPPORTED;
    {
        std::lock_guard<std::mutex> g(g_map_mutex);
        if (g_gate_up_cache.size() >= kMapCacheMax) g_gate_up_cache.clear();
        g_gate_up_cache.emplace(key, GateUpMap{m, sw});
    }
    *map = m;
    *swapped = sw;
    return MOE_OK;
}

// Tile plan.  Rows per expert decide the kernel: with 128 or more on average
// (prefill) the CTA-pair kernel (256 weight rows x token tiles of up to 256
// rows, gemm_pair.cu) keeps the tensor cores fed; with fewer (decode) the
// one-CTA kernel's 128-wide tiles give enough units for every SM to stream
// weights.  An expert never has more than T rows (a token picks an expert at
// most once), so for T <= 128 one row tile of round_up(T, 8) rows holds any
// expert.  The down projection's contraction is split so that enough units
// exist for every SM (one-CTA: about 8 per SM; pairs: about 4 per pair); the
// partial sums are added in the combine.
int make_plan(int T, int d, int ffn, int E, int k, int dt, Plan *p) {
    int rc = check_dims(T, d, ffn, E, k, dt);
    if (rc != MOE_OK) return rc;
    Plan q;
    memset(&q, 0, sizeof q);
    q.T = T;
    q.d = d;
    q.ffn = ffn;
    q.E = E;
    q.k = k;
    q.dt = dt;
    q.rows = T * k;
    q.nchunks = (T + kChunk - 1) / kChunk;
    q.splits = 1;
    q.kps = (ffn + kBlockK - 1) / kBlockK;
    if (dt == MOE_BF16) {
        const long long rows_per_expert = (long long)q.rows / E;
        q.wide = rows_per_expert >= 128 ? 1 : 0;
        // Token tile height of the one-CTA GEMMs: about 1.25x the mean rows
        // per expert, 32, 64, 96 or 128 (and never past the batch): a shorter
        // tile lets the ring hold more weight stages, an expert past it costs
        // one more token tile.  Measured (Mixtral shape, per step): T=100 tile
        // 104 490.0 us, 64 475.4, 32 466.6; T=200 tile 128 502.3, 64 487.3, 32
        // 766.7; T=256 (at most 80 rows an expert) tile 128 495.2, 96 478.5,
        // 64 638.0; T=320 (at most 89) 128 500.3, 96 483.6; T=400 (at most
        // 109) 128 504.0, 96 739.2.
        {
            const long long mu = ((long long)q.rows + E - 1) / E;
            const long long need = (5 * mu + 3) / 4;
            const int tile = need <= 32 ? 32 : need <= 64 ? 64 : need <= 96 ? 96 : 128;
            const int whole = ((T + 7) / 8) * 8;
            q.bm = tile < whole ? tile : whole;
            if (q.bm < 8) q.bm = 8;
        }
        // tuning overrides (measurement only): MOE_PLAN_WIDE=0|1, MOE_PLAN_PAIR=0|1,
        // MOE_PLAN_SPLITS=n, MOE_PLAN_BM=rows (multiple of 8, 8..128)
        if (const char *w = getenv("MOE_PLAN_WIDE")) q.wide = atoi(w) != 0;
        if (const char *b = getenv("MOE_PLAN_BM")) {
            const int v = atoi(b);
            if (v >= 8 && v <= 128 && v % 8 == 0) q.bm = v;
        }
        // many rows per expert: CTA pairs with the tokens as the MMA's N side
        q.pair = q.wide;
        if (const char *pp = getenv("MOE_PLAN_PAIR")) q.pair = atoi(pp) != 0;
        const int kblocks = (ffn + kBlockK - 1) / kBlockK;
        const long long busy = q.rows < E ? q.rows : E;
        long long s = 1;
        const long long smax = kblocks / 8 > 0 ? kblocks / 8 : 1;
        if (q.pair) {
            // down-projection units: 256 features x one token tile of <= 256
            // rows.  No split up to 1024 rows, two below 4 units per pair, none
            // above: the fp32 partial sums cost more than a fuller last wave
            // gains (Mixtral shape, per step, splits 1/2/3/4: T=512 524.3/
            // 538.7/549.9/539.8 us, T=1024 670.4/657.7/683.9/682.9 us, T=2048
            // 1100.9/1098.1/1109.3/1120.2 us)
            const long long ttiles = busy > (q.rows + 255) / 256 ? busy : (q.rows + 255) / 256;
            const long long base_units = ttiles * ((d + 255) / 256);
            s = q.rows <= 1024 ? 1 : base_units >= 4LL * (kPlanSms / 2) ? 1 : 2;
        } else if (!q.wide && busy > 0) {
            // Units: 128 output features x one token tile x one split, for each
            // busy expert.  The split with the least estimated time, in
            // microseconds at about 6.4 TB/s: the busy experts' W2 bytes over
            // the waves of units (a last wave with fewer than 85% of the SMs
            // busy cannot keep HBM saturated, so it costs as if it had 85%),
            // about 0.8 us per unit an SM runs in turn, and the fp32 partial
            // sums (written here, read by the combine: three passes).
            // Busy experts: the expected count under even routing, e = E (1 -
            // (1 - k/E)^T) (exactly k for one token); the cost is weighed
            // between floor(e) and floor(e) + 1 busy experts.  Measured
            // (Mixtral shape, per step): T=1 splits 2 144.7 us, 23 147.6;
            // T=16 splits 1/3/4/5/8 458.3/465.2/452.6/455.7/455.5; T=256
            // splits 1/4 498.5/506.6; T=400 1/4 506.7/522.4.
            const double pk = 1.0 - (double)(k < E ? k : E) / (double)E;
            double ebusy = (double)E * (1.0 - pow(pk, (double)T));
            if (ebusy > (double)busy) ebusy = (double)busy;
            if (ebusy < 1.0) ebusy = 1.0;
            const long long nb_lo = (long long)ebusy;
            const double w_hi = ebusy - (double)nb_lo;
            auto est_us = [&](long long nb, long long c) {
                const long long per_expert = (q.rows + nb - 1) / nb;
                const long long tiles = (per_expert + q.bm - 1) / q.bm;
                const long long units = nb * (tiles > 0 ? tiles : 1) * ((d + 127) / 128) * c;
                const long long waves = (units + kPlanSms - 1) / kPlanSms;
                const double f = (double)(units - (waves - 1) * kPlanSms) / kPlanSms;
                const double t_w = (double)nb * d * ffn * 2 / 6.4e6;
                return t_w * ((double)(waves - 1) + (f > 0.85 ? f : 0.85)) * kPlanSms /
                           (double)units +
                       0.8 * (double)waves + 3.0 * (double)c * q.rows * d * 4 / 6.4e6;
            };
            double best = 1e300;
            for (long long c = 1; c <= smax; ++c) {
                double cost = (1.0 - w_hi) * est_us(nb_lo, c);
                if (w_hi > 0.0) cost += w_hi * est_us(nb_lo + 1, c);
                if (cost < best - 1e-9) {
                    best = cost;
                    s = c;
                }
            }
        }
        if (s > smax) s = smax;
        if (s < 1) s = 1;
        if (const char *sp = getenv("MOE_PLAN_SPLITS")) s = atoi(sp) > 0 ? atoi(sp) : s;
        if (s > kblocks) s = kblocks;
        q.kps = (kblocks + (int)s - 1) / (int)s;
        q.splits = (kblocks + q.kps - 1) / q.kps;
        // The combine folded into the down projection's epilogue: with one
        // split and at most two slots per token, each output element gets at
        // most two fp32 additions into zero, whose sum does not depend on
        // their order.  MOE_FUSE_COMBINE=0|1 forces it off or on where it
        // applies (measurement only).
        q.fuse = (q.pair && q.splits == 1 && k <= 2) ? 1 : 0;
        if (const char *fc = getenv("MOE_FUSE_COMBINE"))
            q.fuse = q.fuse && atoi(fc) != 0;
    }
    const int elt = elem_size(dt);
    // Small batches are grouped by one kernel (counts, scan, ranks and the row
    // copies in one block) instead of two: up to 512 KB of rows to copy (32
    // tokens at hidden 4096 in bf16, top-2), none of them accumulated by the
    // down projection's epilogue (which needs its rows zeroed by the
    // grouping pass).  MOE_ROUTE_SMALL=0|1 forces it where it applies
    // (measurement only).
    {
        const bool fits = (long long)q.rows <= route_small_max();
        q.small_route = fits && (long long)q.rows * d * elt <= (512LL << 10) && !q.fuse;
        if (const char *rs = getenv("MOE_ROUTE_SMALL"))
            q.small_route = fits && !q.fuse && atoi(rs) != 0;
    }
    // The gate/up contraction split in two for the smallest batches (at most
    // 8 expert rows: a few busy experts whose units fill the grid unevenly;
    // the kernel halves them only where that takes fewer rounds), the
    // halves' partial sums added by the later one; the one-kernel grouping
    // zeroes the arrival counters.  Measured (Mixtral shape, per step, whole /
    // halves): T=1 138.2 / 133.3 us, T=4 345.3 / 337.0 us; T=2 and T=3 keep
    // whole units (no fewer rounds).  MOE_PLAN_GSPLIT=0|1 forces it off or on
    // where it applies (measurement only).
    {
        const bool can = dt == MOE_BF16 && !q.wide && !q.pair && q.small_route;
        q.gsplit = can && q.rows <= 8 ? 1 : 0;
        if (const char *gs = getenv("MOE_PLAN_GSPLIT")) q.gsplit = can && atoi(gs) != 0;
        q.nctr = q.gsplit ? ((q.rows + q.bm - 1) / q.bm + E) * ((ffn + 55) / 56) : 0;
    }
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + bytes);
        return o;
    };
    q.o_logits = take((size_t)T * E * 4);
    q.o_idx = take((size_t)T * k * 4);
    q.o_gates = take((size_t)T * k * 4);
    q.o_ccount = take((size_t)q.nchunks * E * 4);
    q.o_cbase = take((size_t)q.nchunks * E * 4);
    q.o_counts = take((size_t)E * 4);
    q.o_offsets = take((size_t)(E + 1) * 4);
    q.o_perm = take((size_t)q.rows * 4);
    q.o_inv = take((size_t)q.rows * 4);
    q.o_rms = take((size_t)T * 4);
    q.o_xperm = take((size_t)q.rows * d * elt);
    q.o_h = take((size_t)q.rows * ffn * elt);
    q.o_y = take((size_t)q.splits * q.rows * d * 4);
    q.o_gpart = take(q.gsplit ? (size_t)2 * q.rows * 2 * ffn * 4 : 0);
    q.o_gctr = take((size_t)q.nctr * 4);
    q.bytes = off;
    *p = q;
    return MOE_OK;
}

namespace {

template <typename T>
T *ws_at(void *ws, size_t off) {
    return reinterpret_cast<T *>(static_cast<uint8_t *>(ws) + off);
}

// Routing options with defaults filled in and checked.
struct Options {
    int gating = MOE_GATING_TOPK_SOFTMAX;
    int capacity = 0;
    int renorm = 0;
};

int read_options(const moe_options *o, Options *out) {
    Options r;
    if (o != nullptr) {
        if (o->gating != MOE_GATING_TOPK_SOFTMAX && o->gating != MOE_GATING_SOFTMAX_TOPK)
            return MOE_ERR_ARG;
        if (o->drop_policy != MOE_DROP_LOSE && o->drop_policy != MOE_DROP_RENORMALIZE)
            return MOE_ERR_ARG;
        r.gating = o->gating;
        r.capacity = o->capacity > 0 ? o->capacity : 0;
        r.renorm = o->drop_policy == MOE_DROP_RENORMALIZE && r.capacity > 0;
    }
    *out = r;
    return MOE_OK;
}

// norm_eps != nullptr: a pre-norm block, out = x (in place):
// x <- round(x + MoE(RMSNorm(x))), RMSNorm fused into the router and the
// grouping, the residual add into the combine.
// x_host_rows != nullptr: the router reads the tokens from page-locked host
// memory (the device's address of it) and copies them to x (device memory)
// for the kernels after it.
int run_forward(const Plan &P, const Options &O, const void *x, const void *W_g,
                const float *bias, const void *const *W1, const void *const *W3,
                const void *const *W2, void *out, void *ws, cudaStream_t s,
                const float *norm_eps = nullptr, const void *x_host_rows = nullptr) {
    float *logits = ws_at<float>(ws, P.o_logits);
    int *idx = ws_at<int>(ws, P.o_idx);
    float *gates = ws_at<float>(ws, P.o_gates);
    int *cc = ws_at<int>(ws, P.o_ccount);
    int *cb = ws_at<int>(ws, P.o_cbase);
    int *counts = ws_at<int>(ws, P.o_counts);
    int *offsets = ws_at<int>(ws, P.o_offsets);
    int *perm = ws_at<int>(ws, P.o_perm);
    int *inv = ws_at<int>(ws, P.o_inv);
    void *x_perm = ws_at<uint8_t>(ws, P.o_xperm);
    void *h = ws_at<uint8_t>(ws, P.o_h);
    float *y = ws_at<float>(ws, P.o_y);
    float *inv_rms = norm_eps != nullptr ? ws_at<float>(ws, P.o_rms) : nullptr;
    const float eps = norm_eps != nullptr ? *norm_eps : 0.f;
    const int elt = elem_size(P.dt);
    // combine in the down projection's epilogue: the fp32 [T][d] accumulator
    // takes the place of y (which holds splits * T * k * d floats)
    const bool fuse = P.fuse && O.capacity == 0;
    int rc;
    if (x_host_rows != nullptr) {
        if ((rc = cuda_rc(launch_router(x_host_rows, W_g, bias, P.T, P.d, P.E, P.k, P.dt,
                                        O.gating, eps, inv_rms, logits, idx, gates, s,
                                        const_cast<void *>(x)))) != MOE_OK)
            return rc;
    } else if ((rc = cuda_rc(launch_router(x, W_g, bias, P.T, P.d, P.E, P.k, P.dt, O.gating, eps,
                                           inv_rms, logits, idx, gates, s))) != MOE_OK) {
        return rc;
    }
    if (P.small_route) {
        if ((rc = cuda_rc(launch_route_small(idx, P.T, P.k, P.E, O.capacity, x, inv_rms, P.d, elt,
                                             counts, offsets, perm, inv, x_perm, s,
                                             P.gsplit ? ws_at<int>(ws, P.o_gctr) : nullptr,
                                             P.nctr))) != MOE_OK)
            return rc;
    } else {
        if ((rc = cuda_rc(launch_chunk_scan(idx, P.T, P.k, P.E, O.capacity, cc, cb, counts,
                                            offsets, s))) != MOE_OK)
            return rc;
        if ((rc = cuda_rc(launch_group_tokens(idx, cb, offsets, x, inv_rms, P.T, P.d, P.E, P.k,
                                              O.capacity, elt, perm, inv, x_perm, s,
                                              fuse ? y : nullptr))) != MOE_OK)
            return rc;
    }
    if (P.dt == MOE_BF16) {
        if (P.pair) {
            if ((rc = launch_swiglu_pair(x_perm, offsets, W1, W3, P.rows, P.d, P.ffn, P.E, h,
                                         s)) != MOE_OK)
                return rc;
            rc = fuse ? launch_down_pair_combine(h, offsets, W2, P.rows, P.d, P.ffn, P.E, perm,
                                                 gates, P.k, y, s)
                      : launch_down_pair(h, offsets, W2, P.rows, P.d, P.ffn, P.E, P.splits,
                                         P.kps, y, s);
            if (rc != MOE_OK) return rc;
        } else {
            if ((rc = launch_swiglu_tc(x_perm, offsets, W1, W3, P.rows, P.d, P.ffn, P.E, P.bm,
                                       P.wide, h, s,
                                       P.gsplit ? ws_at<float>(ws, P.o_gpart) : nullptr,
                                       P.gsplit ? ws_at<int>(ws, P.o_gctr) : nullptr)) != MOE_OK)
                return rc;
            if ((rc = launch_down_tc(h, offsets, W2, P.rows, P.d, P.ffn, P.E, P.bm, P.wide,
                                     P.splits, P.kps, y, s)) != MOE_OK)
                return rc;
        }
    } else {
        if ((rc = cuda_rc(launch_swiglu_f32(static_cast<const float *>(x_perm), offsets, W1, W3,
                                            P.rows, P.d, P.ffn, P.E, static_cast<float *>(h),
                                            s))) != MOE_OK)
            return rc;
        if ((rc = cuda_rc(launch_down_f32(static_cast<const float *>(h), offsets, W2, P.rows, P.d,
                                          P.ffn, P.E, y, s))) != MOE_OK)
            return rc;
    }
    if (fuse)
        return cuda_rc(launch_finalize(y, P.T, P.d, norm_eps != nullptr ? 1 : 0, P.dt, out, s));
    return cuda_rc(launch_combine(y, P.splits, P.rows, gates, inv, P.T, P.d, P.k, O.renorm,
                                  norm_eps != nullptr ? 1 : 0, P.dt, out, s));
}

int check_forward_args(const void *x, const void *W_g, const void *const *W1,
                       const void *const *W3, const void *const *W2, int T, int d, int ffn, int E,
                       int k, int dt, const void *out, const void *ws, size_t ws_bytes,
                       Plan *P) {
    int rc = make_plan(T, d, ffn, E, k, dt, P);
    if (rc != MOE_OK) return rc;
    if ((rc = injected_fault()) != MOE_OK) return rc;
    if (T == 0) return MOE_OK;
    if (x == nullptr || W_g == nullptr || out == nullptr) return MOE_ERR_ARG;
    if ((rc = check_weights(W1, E)) != MOE_OK) return rc;
    if ((rc = check_weights(W3, E)) != MOE_OK) return rc;
    if ((rc = check_weights(W2, E)) != MOE_OK) return rc;
    if (!aligned16(x) || !aligned16(W_g) || !aligned16(out)) return MOE_ERR_UNSUPPORTED;
    if (ws == nullptr || ws_bytes < P->bytes) return MOE_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

// ---- backward ---------------------------------------------------------------

// Scratch of the backward: routing arrays, then row buffers for the padded
// grouping (each expert's block of rows padded to a multiple of 64).
struct BwdPlan {
    int T, d, ffn, E, k, rows, nchunks, nblk;
    size_t o_logits, o_idx, o_gates, o_cc, o_cb, o_counts, o_offsets, o_perm, o_inv, o_gate;
    size_t o_x, o_g, o_U, o_V, o_dU, o_dV, o_gH, o_dgp, o_dx, o_dl, o_part, bytes;
};

int make_bwd_plan(int T, int d, int ffn, int E, int k, int dt, BwdPlan *p) {
    int rc = check_dims(T, d, ffn, E, k, dt);
    if (rc != MOE_OK) return rc;
    if (dt != MOE_BF16) return MOE_ERR_UNSUPPORTED;
    BwdPlan q;
    memset(&q, 0, sizeof q);
    q.T = T;
    q.d = d;
    q.ffn = ffn;
    q.E = E;
    q.k = k;
    q.rows = (T * k + 63) / 64 * 64 + 64 * E;
    q.nchunks = (T + kChunk - 1) / kChunk;
    q.nblk = ffn / 32;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + bytes);
        return o;
    };
    const size_t rows = (size_t)q.rows;
    q.o_logits = take((size_t)T * E * 4);
    q.o_idx = take((size_t)T * k * 4);
    q.o_gates = take((size_t)T * k * 4);
    q.o_cc = take((size_t)q.nchunks * E * 4);
    q.o_cb = take((size_t)q.nchunks * E * 4);
    q.o_counts = take((size_t)E * 4);
    q.o_offsets = take((size_t)(E + 1) * 4);
    q.o_perm = take(rows * 4);
    q.o_inv = take((size_t)T * k * 4);
    q.o_gate = take(rows * 4);
    q.o_x = take(rows * d * 2);
    q.o_g = take(rows * d * 2);
    q.o_U = take(rows * ffn * 2);
    q.o_V = take(rows * ffn * 2);
    q.o_dU = take(rows * ffn * 2);
    q.o_dV = take(rows * ffn * 2);
    q.o_gH = take(rows * ffn * 2);
    q.o_dgp = take(rows * q.nblk * 4);
    q.o_dx = take(rows * d * 4);
    q.o_dl = take((size_t)T * k * 4);
    q.o_part = take(router_wg_part_floats(T, E, d) * 4);
    q.bytes = off;
    *p = q;
    return MOE_OK;
}

// ---- launch graphs -------------------------------------------------------
// A call with the same arguments as an earlier one (every pointer, size,
// option and the plan) replays a CUDA graph of that call's launches: one graph
// launch instead of six kernel launches with parameter blocks of up to 18 KB,
// and the kernels start back to back.  The first call of an argument set runs
// directly (and does the one-time setup: function attributes, the status
// word); the second captures its launches on a private stream (relaxed mode)
// and launches the graph on the caller's stream, as do later calls.  A call on
// a stream that is being captured itself enqueues its kernels directly, so
// they land in the caller's graph.  At most kGraphSlots argument sets are
// kept: a new one takes the place of the one used least recently (its graph
// is destroyed; one still running is freed when it completes).  Counters of
// replays, captures, direct calls and evictions are read with
// moe_graph_cache_stats.  MOE_GRAPHS=0 turns graphs off.
constexpr size_t kGraphSlots = 64;

struct GraphEntry {
    cudaGraphExec_t exec = nullptr;
    bool failed = false;
    unsigned long long last_use = 0;
};

std::mutex g_graph_mutex;
std::unordered_map<std::string, GraphEntry> g_graphs;
cudaStream_t g_capture_stream[64];
unsigned long long g_graph_tick = 0;
moe_graph_stats g_graph_stats = {0, 0, 0, 0, 0};

// Caller holds g_graph_mutex.  Drops the least recently used argument set.
void evict_lru_graph() {
    auto victim = g_graphs.end();
    for (auto it = g_graphs.begin(); it != g_graphs.end(); ++it)
        if (victim == g_graphs.end() || it->second.last_use < victim->second.last_use) victim = it;
    if (victim == g_graphs.end()) return;
    if (victim->second.exec != nullptr) cudaGraphExecDestroy(victim->second.exec);
    g_graphs.erase(victim);
    ++g_graph_stats.evictions;
}

bool graphs_enabled() {
    const char *v = getenv("MOE_GRAPHS");
    return v == nullptr || atoi(v) != 0;
}

// Bytes of every argument that shapes the launches.
class LaunchKey {
  public:
    explicit LaunchKey(int entry) { add(entry); }
    template <typename V>
    LaunchKey &add(const V &v) {
        s_.append(reinterpret_cast<const char *>(&v), sizeof v);
        return *this;
    }
    LaunchKey &ptrs(const void *const *p, int n) {
        for (int i = 0; i < n; ++i) add(p[i]);
        return *this;
    }
    LaunchKey &plan(const Plan &P) {
        return add(P.T).add(P.d).add(P.ffn).add(P.E).add(P.k).add(P.dt).add(P.rows).add(P.wide)
            .add(P.pair).add(P.bm).add(P.splits).add(P.kps).add(P.fuse).add(P.small_route)
            .add(P.gsplit).add(P.bytes);
    }
    LaunchKey &opts(const Options &O) { return add(O.gating).add(O.capacity).add(O.renorm); }
    const std::string &str() const { return s_; }

  private:
    std::string s_;
};

template <typename F>
int run_graphed(const LaunchKey &key, cudaStream_t user, F &&enqueue) {
    auto direct = [&]() {
        {
            std::lock_guard<std::mutex> g(g_graph_mutex);
            ++g_graph_stats.direct_calls;
        }
        return enqueue(user);
    };
    if (!graphs_enabled()) return direct();
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(user, &cs) != cudaSuccess) {
        cudaGetLastError();
        return direct();
    }
    if (cs != cudaStreamCaptureStatusNone) return direct();
    const int dev = current_device();
    if (dev < 0 || dev >= 64) return direct();
    std::string k = key.str();
    k.append(reinterpret_cast<const char *>(&dev), sizeof dev);
    std::lock_guard<std::mutex> g(g_graph_mutex);
    auto it = g_graphs.find(k);
    if (it == g_graphs.end()) {
        if (g_graphs.size() >= kGraphSlots) evict_lru_graph();
        GraphEntry fresh;
        fresh.last_use = ++g_graph_tick;
        g_graphs.emplace(k, fresh);
        ++g_graph_stats.direct_calls;
        return enqueue(user);
    }
    GraphEntry &e = it->second;
    e.last_use = ++g_graph_tick;
    if (e.exec != nullptr) {
        ++g_graph_stats.replays;
        return cudaGraphLaunch(e.exec, user) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
    }
    if (e.failed) {
        ++g_graph_stats.direct_calls;
        return enqueue(user);
    }
    if (g_capture_stream[dev] == nullptr &&
        cudaStreamCreateWithFlags(&g_capture_stream[dev], cudaStreamNonBlocking) != cudaSuccess) {
        g_capture_stream[dev] = nullptr;
        cudaGetLastError();
        e.failed = true;
        ++g_graph_stats.direct_calls;
        return enqueue(user);
    }
    cudaStream_t cap = g_capture_stream[dev];
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    int rc = MOE_ERR_CUDA;
    if (cudaStreamBeginCapture(cap, cudaStreamCaptureModeRelaxed) == cudaSuccess) {
        rc = enqueue(cap);
        if (cudaStreamEndCapture(cap, &graph) != cudaSuccess) graph = nullptr;
    }
    if (rc == MOE_OK && graph != nullptr && cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess)
        exec = nullptr;
    if (graph != nullptr) cudaGraphDestroy(graph);
    if (exec == nullptr) {
        cudaGetLastError();
        e.failed = true;
        ++g_graph_stats.direct_calls;
        return enqueue(user);
    }
    e.exec = exec;
    ++g_graph_stats.captures;
    return cudaGraphLaunch(exec, user) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

LaunchKey forward_key(int entry, const Plan &P, const Options &O, const void *x,
                      const void *W_g, const float *bias, const void *const *W1,
                      const void *const *W3, const void *const *W2, const void *out,
                      const void *ws) {
    LaunchKey key(entry);
    key.plan(P).opts(O).add(x).add(W_g).add(bias).ptrs(W1, P.E).ptrs(W3, P.E).ptrs(W2, P.E)
        .add(out).add(ws);
    return key;
}

int run_backward(const BwdPlan &P, const void *x, const void *W_g, const float *bias,
                 const void *const *W1, const void *const *W3, const void *const *W2,
                 const void *d_out, void *d_x, float *d_Wg, float *const *d_W1,
                 float *const *d_W3, float *const *d_W2, void *ws, cudaStream_t s) {
    const int T = P.T, d = P.d, ffn = P.ffn, E = P.E, k = P.k, rows = P.rows;
    float *logits = ws_at<float>(ws, P.o_logits);
    int *idx = ws_at<int>(ws, P.o_idx);
    float *gates = ws_at<float>(ws, P.o_gates);
    int *cc = ws_at<int>(ws, P.o_cc);
    int *cb = ws_at<int>(ws, P.o_cb);
    int *counts = ws_at<int>(ws, P.o_counts);
    int *offsets = ws_at<int>(ws, P.o_offsets);
    int *perm = ws_at<int>(ws, P.o_perm);
    int *inv = ws_at<int>(ws, P.o_inv);
    float *row_gate = ws_at<float>(ws, P.o_gate);
    void *x_rows = ws_at<uint8_t>(ws, P.o_x);
    void *g_rows = ws_at<uint8_t>(ws, P.o_g);
    void *U = ws_at<uint8_t>(ws, P.o_U);
    void *V = ws_at<uint8_t>(ws, P.o_V);
    void *dU = ws_at<uint8_t>(ws, P.o_dU);
    void *dV = ws_at<uint8_t>(ws, P.o_dV);
    void *gH = ws_at<uint8_t>(ws, P.o_gH);
    float *dgp = ws_at<float>(ws, P.o_dgp);
    float *dx_rows = ws_at<float>(ws, P.o_dx);
    float *dl = ws_at<float>(ws, P.o_dl);
    float *part = ws_at<float>(ws, P.o_part);
    int rc;
    // routing again, grouped with each expert's rows padded to 64
    if ((rc = cuda_rc(launch_router(x, W_g, bias, T, d, E, k, MOE_BF16, MOE_GATING_TOPK_SOFTMAX,
                                    0.f, nullptr, logits, idx, gates, s))) != MOE_OK)
        return rc;
    if ((rc = cuda_rc(launch_chunk_scan(idx, T, k, E, 0, cc, cb, counts, offsets, s, 64))) !=
        MOE_OK)
        return rc;
    if ((rc = cuda_rc(cudaMemsetAsync(perm, 0xFF, (size_t)rows * 4, s))) != MOE_OK) return rc;
    if ((rc = cuda_rc(launch_group_tokens(idx, cb, offsets, nullptr, nullptr, T, 0, E, k, 0, 0,
                                          perm, inv, nullptr, s))) != MOE_OK)
        return rc;
    if ((rc = cuda_rc(launch_gather_rows(x, perm, offsets, E, rows, k, d, nullptr, nullptr,
                                         x_rows, s))) != MOE_OK)
        return rc;
    if ((rc = cuda_rc(launch_gather_rows(d_out, perm, offsets, E, rows, k, d, gates, row_gate,
                                         g_rows, s))) != MOE_OK)
        return rc;
    // expert GEMMs
    if ((rc = launch_bwd_uv(x_rows, offsets, W1, W3, rows, d, ffn, E, U, V, s)) != MOE_OK)
        return rc;
    if ((rc = launch_bwd_z(g_rows, offsets, W2, rows, d, ffn, E, U, V, row_gate, dU, dV, gH, dgp,
                           s)) != MOE_OK)
        return rc;
    if ((rc = launch_bwd_dx(dU, dV, offsets, W1, W3, rows, d, ffn, E, dx_rows, s)) != MOE_OK)
        return rc;
    if ((rc = launch_bwd_wgrad(x_rows, g_rows, dU, dV, gH, offsets, rows, d, ffn, E, d_W1, d_W3,
                               d_W2, s)) != MOE_OK)
        return rc;
    // router and input gradients
    if ((rc = cuda_rc(launch_router_bwd(idx, gates, inv, dgp, P.nblk, dx_rows, W_g, T, d, k, dl,
                                        d_x, s))) != MOE_OK)
        return rc;
    return cuda_rc(launch_router_wgrad(idx, dl, x, T, d, E, k, part, d_Wg, s));
}

}  // namespace

// The layer with its kernels enqueued directly on `s`: validation, plan and
// the launch sequence of moe_forward, without the launch-graph cache (so no
// stream or graph is created on the way).
int forward_direct(const void *x, const void *W_g, const float *router_bias,
                   const void *const *W1, const void *const *W3, const void *const *W2, int T,
                   int d, int ffn, int E, int k, int dtype, void *out, void *workspace,
                   size_t workspace_bytes, cudaStream_t s) {
    Plan P;
    int rc = check_forward_args(x, W_g, W1, W3, W2, T, d, ffn, E, k, dtype, out, workspace,
                                workspace_bytes, &P);
    if (rc != MOE_OK || T == 0) return rc;
    return run_forward(P, Options(), x, W_g, router_bias, W1, W3, W2, out, workspace, s);
}

}  // namespace moe

using namespace moe;

extern "C" {

const char *moe_strerror(int status) {
    switch (status) {
        case MOE_OK: return "ok";
        case MOE_ERR_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported shape, type or alignment";
        case MOE_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
        case MOE_ERR_CUDA: return "CUDA runtime or launch error";
        case MOE_ERR_DEVICE: return "a kernel's bounded wait expired";
        default: return "unknown status";
    }
}

int moe_version(void) { return 100; }

int moe_workspace_bytes(int T, int d, int ffn, int E, int k, int dtype, size_t *bytes) {
    if (bytes == nullptr) return MOE_ERR_ARG;
    Plan P;
    const int rc = make_plan(T, d, ffn, E, k, dtype, &P);
    if (rc != MOE_OK) return rc;
    *bytes = P.bytes;
    return MOE_OK;
}

int moe_backward_workspace_bytes(int T, int d, int ffn, int E, int k, int dtype, size_t *bytes) {
    if (bytes == nullptr) return MOE_ERR_ARG;
    BwdPlan P;
    const int rc = make_bwd_plan(T, d, ffn, E, k, dtype, &P);
    if (rc != MOE_OK) return rc;
    *bytes = P.bytes;
    return MOE_OK;
}

int moe_backward(const void *x, const void *W_g, const float *router_bias, const void *const *W1,
                 const void *const *W3, const void *const *W2, int T, int d, int ffn, int E, int k,
                 int dtype, const void *d_out, void *d_x, float *d_W_g, float *const *d_W1,
                 float *const *d_W3, float *const *d_W2, void *workspace, size_t workspace_bytes,
                 void *stream) {
    BwdPlan P;
    int rc = make_bwd_plan(T, d, ffn, E, k, dtype, &P);
    if (rc != MOE_OK) return rc;
    if ((rc = injected_fault()) != MOE_OK) return rc;
    if (W_g == nullptr || d_W_g == nullptr || d_W1 == nullptr || d_W3 == nullptr ||
        d_W2 == nullptr)
        return MOE_ERR_ARG;
    if ((rc = check_weights(W1, E)) != MOE_OK) return rc;
    if ((rc = check_weights(W3, E)) != MOE_OK) return rc;
    if ((rc = check_weights(W2, E)) != MOE_OK) return rc;
    for (int e = 0; e < E; ++e)
        if (d_W1[e] == nullptr || d_W3[e] == nullptr || d_W2[e] == nullptr)
            return MOE_ERR_ARG;
    for (int e = 0; e < E; ++e)
        if (!aligned16(d_W1[e]) || !aligned16(d_W3[e]) || !aligned16(d_W2[e]))
            return MOE_ERR_UNSUPPORTED;
    if (!aligned16(W_g) || !aligned16(d_W_g)) return MOE_ERR_UNSUPPORTED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T == 0) {
        // no tokens: every gradient is zero
        if (cudaMemsetAsync(d_W_g, 0, sizeof(float) * E * d, s) != cudaSuccess) return MOE_ERR_CUDA;
        for (int e = 0; e < E; ++e) {
            const size_t n = sizeof(float) * (size_t)ffn * d;
            if (cudaMemsetAsync(d_W1[e], 0, n, s) != cudaSuccess ||
                cudaMemsetAsync(d_W3[e], 0, n, s) != cudaSuccess ||
                cudaMemsetAsync(d_W2[e], 0, n, s) != cudaSuccess)
                return MOE_ERR_CUDA;
        }
        return MOE_OK;
    }
    if (x == nullptr || d_out == nullptr || d_x == nullptr) return MOE_ERR_ARG;
    if (!aligned16(x) || !aligned16(d_out) || !aligned16(d_x)) return MOE_ERR_UNSUPPORTED;
    if (workspace == nullptr || workspace_bytes < P.bytes) return MOE_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return MOE_ERR_WORKSPACE;
    return run_backward(P, x, W_g, router_bias, W1, W3, W2, d_out, d_x, d_W_g, d_W1, d_W3, d_W2,
                        workspace, s);
}

int moe_forward_launches(int T, int d, int ffn, int E, int k, int dtype, int *launches) {
    if (launches == nullptr) return MOE_ERR_ARG;
    Plan P;
    const int rc = make_plan(T, d, ffn, E, k, dtype, &P);
    if (rc != MOE_OK) return rc;
    // router, scan + group (one kernel for small batches), gate/up, down,
    // combine (or the finalize of the combine folded into the down projection)
    *launches = T == 0 ? 0 : (P.small_route ? 5 : 6);
    return MOE_OK;
}

int moe_graph_cache_stats(moe_graph_stats *stats, int reset) {
    if (stats == nullptr) return MOE_ERR_ARG;
    std::lock_guard<std::mutex> g(g_graph_mutex);
    *stats = g_graph_stats;
    stats->entries = static_cast<long long>(g_graphs.size());
    if (reset) g_graph_stats = moe_graph_stats{0, 0, 0, 0, 0};
    return MOE_OK;
}

int moe_down_splits(int T, int d, int ffn, int E, int k, int dtype, int *splits) {
    if (splits == nullptr) return MOE_ERR_ARG;
    Plan P;
    const int rc = make_plan(T, d, ffn, E, k, dtype, &P);
    if (rc != MOE_OK) return rc;
    *splits = P.splits;
    return MOE_OK;
}

int moe_forward(const void *x, const void *W_g, const float *router_bias, const void *const *W1,
                const void *const *W3, const void *const *W2, int T, int d, int ffn, int E, int k,
                int dtype, void *out, void *workspace, size_t workspace_bytes, void *stream) {
    Plan P;
    int rc = check_forward_args(x, W_g, W1, W3, W2, T, d, ffn, E, k, dtype, out, workspace,
                                workspace_bytes, &P);
    if (rc != MOE_OK || T == 0) return rc;
    const Options O;
    return run_graphed(forward_key(1, P, O, x, W_g, router_bias, W1, W3, W2, out, workspace),
                       static_cast<cudaStream_t>(stream), [&](cudaStream_t s) {
                           return run_forward(P, O, x, W_g, router_bias, W1, W3, W2, out,
                                              workspace, s);
                       });
}

int moe_forward_ex(const void *x, const void *W_g, const float *router_bias,
                   const void *const *W1, const void *const *W3, const void *const *W2, int T,
                   int d, int ffn, int E, int k, int dtype, const moe_options *options, void *out,
                   void *workspace, size_t workspace_bytes, void *stream) {
    Options O;
    int rc = read_options(options, &O);
    if (rc != MOE_OK) return rc;
    Plan P;
    rc = check_forward_args(x, W_g, W1, W3, W2, T, d, ffn, E, k, dtype, out, workspace,
                            workspace_bytes, &P);
    if (rc != MOE_OK || T == 0) return rc;
    return run_graphed(forward_key(2, P, O, x, W_g, router_bias, W1, W3, W2, out, workspace),
                       static_cast<cudaStream_t>(stream), [&](cudaStream_t s) {
                           return run_forward(P, O, x, W_g, router_bias, W1, W3, W2, out,
                                              workspace, s);
                       });
}

int moe_block_forward(void *x, const void *W_g, const float *router_bias, const void *const *W1,
                      const void *const *W3, const void *const *W2, int T, int d, int ffn, int E,
                      int k, int dtype, float eps, const moe_options *options, void *workspace,
                      size_t workspace_bytes, void *stream) {
    if (!(eps >= 0.f)) return MOE_ERR_ARG;
    Options O;
    int rc = read_options(options, &O);
    if (rc != MOE_OK) return rc;
    Plan P;
    rc = check_forward_args(x, W_g, W1, W3, W2, T, d, ffn, E, k, dtype, x, workspace,
                            workspace_bytes, &P);
    if (rc != MOE_OK || T == 0) return rc;
    LaunchKey key = forward_key(3, P, O, x, W_g, router_bias, W1, W3, W2, x, workspace);
    key.add(eps);
    return run_graphed(key, static_cast<cudaStream_t>(stream), [&](cudaStream_t s) {
        return run_forward(P, O, x, W_g, router_bias, W1, W3, W2, x, workspace, s, &eps);
    });
}

int moe_capacity(double capacity_factor, int T, int k, int E, int *capacity) {
    if (capacity == nullptr || T < 0 || k < 1 || E < 1) return MOE_ERR_ARG;
    if (!(capacity_factor > 0.0)) {
        *capacity = 0;
        return MOE_OK;
    }
    const double c = ceil(capacity_factor * (double)T * (double)k / (double)E);
    if (c > 2147483647.0) return MOE_ERR_ARG;
    *capacity = (int)c;
    return MOE_OK;
}

namespace {

// The device's address for page-locked (pinned or registered) host memory,
// or nullptr for any other pointer (pageable memory, device memory).
void *device_alias_of_host(const void *p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (at.type != cudaMemoryTypeHost || at.devicePointer == nullptr) return nullptr;
    return at.devicePointer;
}

}  // namespace

int moe_forward_host_io(const void *x_host, void *out_host, void *x_dev, void *out_dev,
                        const void *W_g, const float *router_bias, const void *const *W1,
                        const void *const *W3, const void *const *W2, int T, int d, int ffn,
                        int E, int k, int dtype, void *workspace, size_t workspace_bytes,
                        void *stream) {
    Plan P;
    int rc = check_forward_args(x_dev, W_g, W1, W3, W2, T, d, ffn, E, k, dtype, out_dev,
                                workspace, workspace_bytes, &P);
    if (rc != MOE_OK || T == 0) return rc;
    if (x_host == nullptr || out_host == nullptr) return MOE_ERR_ARG;
    const size_t bytes = (size_t)T * d * elem_size(dtype);
    const Options O;
    // A page-locked out_host is written by the layer's last kernel directly
    // (no device-to-host copy; out_dev is then not touched).  For batches the
    // router takes in one pass, a page-locked x_host is read by the router
    // itself, which leaves the rows in x_dev for the later kernels (no
    // host-to-device copy).  MOE_HOSTIO_DIRECT=0 keeps both copies
    // (measurement only).
    void *out_alias = nullptr;
    const void *x_alias = nullptr;
    {
        const char *v = getenv("MOE_HOSTIO_DIRECT");
        if (v == nullptr || atoi(v) != 0) {
            out_alias = device_alias_of_host(out_host);
            if (out_alias != nullptr && !aligned16(out_alias)) out_alias = nullptr;
            if (dtype == MOE_BF16 && router_reads_host_rows(T, E)) {
                x_alias = device_alias_of_host(x_host);
                if (x_alias != nullptr && !aligned16(x_alias)) x_alias = nullptr;
            }
        }
    }
    LaunchKey key = forward_key(4, P, O, x_dev, W_g, router_bias, W1, W3, W2, out_dev, workspace);
    key.add(x_host).add(out_host).add(out_alias).add(x_alias);
    return run_graphed(key, static_cast<cudaStream_t>(stream), [&](cudaStream_t s) {
        if (x_alias == nullptr &&
            cudaMemcpyAsync(x_dev, x_host, bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
            return (int)MOE_ERR_CUDA;
        int r = run_forward(P, O, x_dev, W_g, router_bias, W1, W3, W2,
                            out_alias != nullptr ? out_alias : out_dev, workspace, s, nullptr,
                            x_alias);
        if (r != MOE_OK) return r;
        if (out_alias == nullptr &&
            cudaMemcpyAsync(out_host, out_dev, bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
            return (int)MOE_ERR_CUDA;
        return (int)MOE_OK;
    });
}

int moe_router(const void *x, const void *W_g, const float *router_bias, int T, int d, int E,
               int k, int dtype, float *logits, int *idx, float *gates, void *stream) {
    int rc = check_dims(T, d, 64, E, k, dtype);
    if (rc != MOE_OK) return rc;
    if ((rc = injected_fault()) != MOE_OK) return rc;
    if (T == 0) return MOE_OK;
    if (!x || !W_g || !logits || !idx || !gates) return MOE_ERR_ARG;
    if (!aligned16(x) || !aligned16(W_g)) return MOE_ERR_UNSUPPORTED;
    return cuda_rc(launch_router(x, W_g, router_bias, T, d, E, k, dtype, MOE_GATING_TOPK_SOFTMAX,
                                 0.f, nullptr, logits, idx, gates,
                                 static_cast<cudaStream_t>(stream)));
}

int moe_route_workspace_bytes(int T, int E, int k, size_t *bytes) {
    if (bytes == nullptr) return MOE_ERR_ARG;
    int rc = check_dims(T, 64, 64, E, k, MOE_BF16);
    if (rc != MOE_OK) return rc;
    const size_t nchunks = (size_t)(T + kChunk - 1) / kChunk;
    *bytes = 2 * align_up(nchunks * E * 4);
    return MOE_OK;
}

int moe_route_from_logits(const float *logits, int T, int E, int k, int *idx, float *gates,
                          int *counts, int *offsets, int *perm, int *inv, void *workspace,
                          size_t workspace_bytes, void *stream) {
    return moe_route_from_logits_ex(logits, T, E, k, nullptr, idx, gates, counts, offsets, perm,
                                    inv, workspace, workspace_bytes, stream);
}

int moe_route_from_logits_ex(const float *logits, int T, int E, int k,
                             const moe_options *options, int *idx, float *gates, int *counts,
                             int *offsets, int *perm, int *inv, void *workspace,
                             size_t workspace_bytes, void *stream) {
    Options O;
    int rc = read_options(options, &O);
    if (rc != MOE_OK) return rc;
    rc = check_dims(T, 64, 64, E, k, MOE_BF16);
    if (rc != MOE_OK) return rc;
    if ((rc = injected_fault()) != MOE_OK) return rc;
    if (!counts || !offsets) return MOE_ERR_ARG;
    size_t need = 0;
    moe_route_workspace_bytes(T, E, k, &need);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T == 0) {
        // no rows: every count is zero and every offset is zero
        if (cudaMemsetAsync(counts, 0, (size_t)E * 4, s) != cudaSuccess) return MOE_ERR_CUDA;
        if (cudaMemsetAsync(offsets, 0, (size_t)(E + 1) * 4, s) != cudaSuccess)
            return MOE_ERR_CUDA;
        return MOE_OK;
    }
    if (!logits || !idx || !gates || !perm || !inv) return MOE_ERR_ARG;
    if (workspace == nullptr || workspace_bytes < need) return MOE_ERR_WORKSPACE;
    const int nchunks = (T + kChunk - 1) / kChunk;
    int *cc = static_cast<int *>(workspace);
    int *cb = reinterpret_cast<int *>(static_cast<uint8_t *>(workspace) +
                                      align_up((size_t)nchunks * E * 4));
    if ((rc = cuda_rc(launch_topk_from_logits(logits, T, E, k, O.gating, idx, gates, s))) !=
        MOE_OK)
        return rc;
    if ((rc = cuda_rc(launch_chunk_scan(idx, T, k, E, O.capacity, cc, cb, counts, offsets, s))) !=
        MOE_OK)
        return rc;
    return cuda_rc(launch_group_tokens(idx, cb, offsets, nullptr, nullptr, T, 0, E, k, O.capacity,
                                       0, perm, inv, nullptr, s));
}

int moe_permute(const void *x, const int *perm, int rows, int T, int d, int k, int dtype,
                void *x_perm, void *stream) {
    int rc = check_dims(T, d, 64, k, k, dtype);
    if (rc != MOE_OK) return rc;
    if (rows < 0 || (long long)rows > (long long)T * k) return MOE_ERR_ARG;
    if (rows == 0) return MOE_OK;
    if (!x || !perm || !x_perm) return MOE_ERR_ARG;
    if (!aligned16(x) || !aligned16(x_perm)) return MOE_ERR_UNSUPPORTED;
    return cuda_rc(launch_permute(x, perm, rows, d, k, elem_size(dtype), x_perm,
                                  static_cast<cudaStream_t>(stream)));
}

int moe_expert_swiglu(const void *x_perm, const int *offsets, const void *const *W1,
                      const void *const *W3, int rows, int d, int ffn, int E, int dtype, void *h,
                      void *stream) {
    int rc = check_dims(rows, d, ffn, E, 1, dtype);
    if (rc != MOE_OK) return rc;
    if ((rc = injected_fault()) != MOE_OK) return rc;
    if (rows == 0) return MOE_OK;
    if (!x_perm || !offsets || !h) return MOE_ERR_ARG;
    if ((rc = check_weights(W1, E)) != MOE_OK) return rc;
    if ((rc = check_weights(W3, E)) != MOE_OK) return rc;
    if (!aligned16(x_perm) || !aligned16(h)) return MOE_ERR_UNSUPPORTED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == MOE_BF16) {
        // plan as if the rows came from T = rows / 2 tokens with k = 2 when
        // possible, else one token per row
        Plan P;
        const int k = (rows % 2 == 0 && E >= 2) ? 2 : 1;
        if ((rc = make_plan(rows / k, d, ffn, E, k, dtype, &P)) != MOE_OK) return rc;
        if (P.pair) return launch_swiglu_pair(x_perm, offsets, W1, W3, rows, d, ffn, E, h, s);
        return launch_swiglu_tc(x_perm, offsets, W1, W3, rows, d, ffn, E, P.bm, P.wide, h, s);
    }
    return cuda_rc(launch_swiglu_f32(static_cast<const float *>(x_perm), offsets, W1, W3, rows, d,
                                     ffn, E, static_cast<float *>(h), s));
}

int moe_expert_down(const void *h, const int *offsets, const void *const *W2, int T, int d,
                    int ffn, int E, int k, int dtype, float *y_partial, void *stream) {
    Plan P;
    int rc = make_plan(T, d, ffn, E, k, dtype, &P);
    if (rc != MOE_OK) return rc;
    if ((rc = injected_fault()) != MOE_OK) return rc;
    if (T == 0) return MOE_OK;
    if (!h || !offsets || !y_partial) return MOE_ERR_ARG;
    if ((rc = check_weights(W2, E)) != MOE_OK) return rc;
    if (!aligned16(h) || !aligned16(y_partial)) return MOE_ERR_UNSUPPORTED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == MOE_BF16)
        return P.pair ? launch_down_pair(h, offsets, W2, P.rows, d, ffn, E, P.splits, P.kps,
                                         y_partial, s)
                      : launch_down_tc(h, offsets, W2, P.rows, d, ffn, E, P.bm, P.wide, P.splits,
                                       P.kps, y_partial, s);
    return cuda_rc(launch_down_f32(static_cast<const float *>(h), offsets, W2, P.rows, d, ffn, E,
                                   y_partial, s));
}

int moe_combine(const float *y_partial, int splits, const float *gates, const int *inv, int T,
                int d, int k, int dtype, void *out, void *stream) {
    int rc = check_dims(T, d, 64, k, k, dtype);
    if (rc != MOE_OK) return rc;
    if (splits < 1) return MOE_ERR_ARG;
    if (T == 0) return MOE_OK;
    if (!y_partial || !gates || !inv || !out) return MOE_ERR_ARG;
    if (d % 4 != 0 || !aligned16(y_partial) || !aligned16(out)) return MOE_ERR_UNSUPPORTED;
    return cuda_rc(launch_combine(y_partial, splits, T * k, gates, inv, T, d, k, 0, 0, dtype, out,
                                  static_cast<cudaStream_t>(stream)));
}

int moe_add_rmsnorm(void *x, const void *add, void *xn, int T, int d, float eps, int dtype,
                    void *stream) {
    if (T < 0 || d <= 0 || (dtype != MOE_F32 && dtype != MOE_BF16) || !(eps >= 0.f))
        return MOE_ERR_ARG;
    if (T == 0) return MOE_OK;
    if (!x || !xn) return MOE_ERR_ARG;
    if ((d * elem_size(dtype)) % 16 != 0 || !aligned16(x) || !aligned16(xn) ||
        (add != nullptr && !aligned16(add)))
        return MOE_ERR_UNSUPPORTED;
    return cuda_rc(launch_add_rmsnorm(x, add, xn, T, d, eps, dtype,
                                      static_cast<cudaStream_t>(stream)));
}

int moe_device_status(void *stream, int *status, int clear) {
    if (status == nullptr) return MOE_ERR_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof v) != cudaSuccess) return MOE_ERR_CUDA;
    *status = v;
    if (clear && v != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_device_status, &zero, sizeof zero) != cudaSuccess)
            return MOE_ERR_CUDA;
    }
    return MOE_OK;
}

int moe_selftest_wait_timeout(unsigned int limit_ns, void *stream) {
    if (limit_ns < 1000u) limit_ns = 1000u;
    if (limit_ns > 100000000u) limit_ns = 100000000u;
    return cuda_rc(launch_wait_selftest(limit_ns, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
