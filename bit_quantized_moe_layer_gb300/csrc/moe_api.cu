// C ABI of libmoe (declared in include/moe.h): argument checks, workspace
// layout, TMA descriptors and the launch sequence of the routed 4-bit MoE
// layer (DiffRouter + DiffExperts of "diffusion-gemma/model.ts").
//
// All checks happen on the host before anything is enqueued; the CUDA
// runtime is touched only after the arguments passed, so the checks work on
// a machine without a GPU.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "../../include/moe.h"
#include "kernels.h"

using namespace moe;

namespace {

constexpr int kStages = 6;  // route, dispatch, gather, gate_up, down, combine
constexpr int kMaxTimedCalls = 1024;

// --------------------------------------------------------------- checks --
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_dims(const moe_dims* d) {
    if (!d) return MOE_ERR_NULL;
    if (d->T < 0 || d->H <= 0 || d->E <= 0 || d->k <= 0 || d->inter <= 0) return MOE_ERR_SHAPE;
    if (d->bits != 4 || d->group != 64) return MOE_ERR_UNSUPPORTED;
    if (d->H % 128 != 0 || d->inter % 64 != 0 || d->H > 5504) return MOE_ERR_UNSUPPORTED;
    if (d->k > 32 || d->k > d->E || d->E > 256) return MOE_ERR_UNSUPPORTED;
    if ((int64_t)d->T * d->k > (int64_t)1 << 28) return MOE_ERR_SHAPE;
    if (!(d->eps >= 0.0f) || isinf(d->eps)) return MOE_ERR_SHAPE;
    return MOE_OK;
}

int check_ptrs(std::initializer_list<const void*> ps) {
    for (const void* p : ps)
        if (!p) return MOE_ERR_NULL;
    for (const void* p : ps)
        if (!aligned16(p)) return MOE_ERR_ALIGN;
    return MOE_OK;
}

int check_qweight(const moe_qweight* q) {
    if (!q) return MOE_ERR_NULL;
    return check_ptrs({q->w, q->scales, q->biases});
}

// --------------------------------------------------------------- device --
struct DeviceInfo {
    int sms = 0;
    bool ok = false;
};

int device_info(DeviceInfo* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_DEVICE;
    static std::mutex mu;
    static std::vector<DeviceInfo> cache;
    std::lock_guard<std::mutex> lock(mu);
    if ((int)cache.size() <= dev) cache.resize(dev + 1);
    if (!cache[dev].ok) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return MOE_ERR_DEVICE;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MOE_ERR_DEVICE;
        // The library is built for sm_103a only (arch-specific code runs on
        // compute capability 10.3 and nothing else): refuse other GPUs here.
        if (major != 10 || minor != 3) return MOE_ERR_DEVICE;
        cache[dev].sms = sms;
        cache[dev].ok = true;
    }
    *out = cache[dev];
    return MOE_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// A tensor map is a pure function of its encode arguments (address, type,
// sizes, strides, box; the rest is fixed here), so encoded maps are kept in
// a small least-recently-used table: repeated calls on the same buffers (a
// decode or serving loop) skip the ~14 host-side encodes a forward needs.
struct MapKey {
    const void* ptr;
    int dt, rank;
    uint64_t dims[3], strides[2];
    uint32_t box[3];
    bool operator==(const MapKey& o) const {
        if (ptr != o.ptr || dt != o.dt || rank != o.rank) return false;
        for (int i = 0; i < rank; ++i)
            if (dims[i] != o.dims[i] || box[i] != o.box[i]) return false;
        for (int i = 0; i + 1 < rank; ++i)
            if (strides[i] != o.strides[i]) return false;
        return true;
    }
};

bool encode_cached(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* ptr, const uint64_t* dims,
                   const uint64_t* strides, const uint32_t* box) {
    constexpr int kSlots = 64;
    struct Entry {
        MapKey key;
        CUtensorMap map;
        uint64_t used;
    };
    static Entry table[kSlots];
    static uint64_t tick = 0;
    static std::mutex mu;
    MapKey key{ptr, (int)dt, rank, {0, 0, 0}, {0, 0}, {0, 0, 0}};
    for (int i = 0; i < rank; ++i) {
        key.dims[i] = dims[i];
        key.box[i] = box[i];
    }
    for (int i = 0; i + 1 < rank; ++i) key.strides[i] = strides[i];
    {
        std::lock_guard<std::mutex> lock(mu);
        for (Entry& e : table)
            if (e.used && e.key == key) {
                e.used = ++tick;
                *m = e.map;
                return true;
            }
    }
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t d[3], st[2];
    cuuint32_t b[3], estr[3] = {1, 1, 1};
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
    }
    for (int i = 0; i + 1 < rank; ++i) st[i] = strides[i];
    if (fn(m, dt, (cuuint32_t)rank, const_cast<void*>(ptr), d, st, b, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    std::lock_guard<std::mutex> lock(mu);
    Entry* victim = &table[0];
    for (Entry& e : table)
        if (e.used < victim->used) victim = &e;
    victim->key = key;
    victim->map = *m;
    victim->used = ++tick;
    return true;
}

bool make_map_2d(CUtensorMap* m, CUtensorMapDataType dt, size_t esize, const void* ptr, uint64_t inner,
                 uint64_t rows, uint32_t box_inner, uint32_t box_rows) {
    const uint64_t dims[2] = {inner, rows}, strides[1] = {inner * esize};
    const uint32_t box[2] = {box_inner, box_rows};
    return encode_cached(m, dt, 2, ptr, dims, strides, box);
}

// The grouped GEMM's token-operand maps over a bf16 [rows, K] buffer (see
// BMaps): 3-D boxes of 16, 32, 64 and 128 rows by min(4, K/64) atoms, and the
// 2-D 16-row box.
bool make_bmaps(BMaps* b, const void* ptr, uint64_t K, uint64_t rows) {
    if (!make_map_2d(&b->m2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, K, rows, 64, 16)) return false;
    for (int i = 0; i < 4; ++i) {
        const uint64_t dims[3] = {64, rows, K / 64}, strides[2] = {K * 2, 128};
        const uint32_t box[3] = {64, (uint32_t)(16 << i), (uint32_t)(K / 64 < 4 ? K / 64 : 4)};
        if (!encode_cached(&b->m[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ptr, dims, strides, box)) return false;
    }
    return true;
}

// bf16(x) of a double, one rounding to nearest even (x > 0, normal range).
float bf16_round(double x) {
    int e;
    frexp(x, &e);
    const double q = ldexp(1.0, e - 8);
    return (float)(nearbyint(x / q) * q);
}

// ------------------------------------------------------------ workspace --
struct Layout {
    size_t idx, w, perm, inv, offsets, tiles, ntiles, dhist, xs, mid, y, xdev, outdev, total;
    int max_tiles;
};

size_t up256(size_t v) { return (v + 255) & ~size_t(255); }

Layout layout(const moe_dims* d) {
    Layout L;
    const size_t S = (size_t)d->T * d->k;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        size_t at = o;
        o = up256(o + (bytes ? bytes : 1));
        return at;
    };
    L.max_tiles = d->E + (int)((S + kGemvRows - 1) / kGemvRows);  // token tiles of >= kGemvRows rows
    L.idx = take(S * 4);
    L.w = take(S * 2);
    L.perm = take(S * 4);
    L.inv = take(S * 4);
    L.offsets = take((size_t)(d->E + 1) * 4);
    L.tiles = take((size_t)L.max_tiles * sizeof(Tile));
    L.ntiles = take(8);
    L.dhist = take((size_t)kDispatchMaxChunks * d->E * 4);
    L.xs = take(S * d->H * 2);
    L.mid = take(S * d->inter * 2);
    L.y = take(S * d->H * 2);
    L.xdev = take((size_t)d->T * d->H * 2);  // host-I/O input, or the branch's expert input
    L.outdev = take((size_t)d->T * d->H * 2);
    L.total = o;
    return L;
}

// Library-owned grow-only workspace, one per device.
int owned_workspace(size_t bytes, void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_DEVICE;
    static std::mutex mu;
    static std::vector<std::pair<void*, size_t>> bufs;
    std::lock_guard<std::mutex> lock(mu);
    if ((int)bufs.size() <= dev) bufs.resize(dev + 1, {nullptr, 0});
    if (bufs[dev].second < bytes) {
        if (bufs[dev].first) {
            cudaDeviceSynchronize();
            cudaFree(bufs[dev].first);
        }
        bufs[dev] = {nullptr, 0};
        void* p = nullptr;
        if (cudaMalloc(&p, bytes) != cudaSuccess) return MOE_ERR_CUDA;
        bufs[dev] = {p, bytes};
    }
    *out = bufs[dev].first;
    return MOE_OK;
}

// --------------------------------------------------------------- timing --
struct Timing {
    bool enabled = false;
    std::vector<cudaEvent_t> ev;  // kMaxTimedCalls * (kStages + 1)
    int calls = 0;
    std::mutex mu;
};
Timing& timing() {
    static Timing t;
    return t;
}

// Records boundary b (0..kStages) of the current timed call, if any.
struct CallTimer {
    cudaEvent_t* ev = nullptr;
    cudaStream_t s;
    explicit CallTimer(cudaStream_t st) : s(st) {
        Timing& t = timing();
        std::lock_guard<std::mutex> lock(t.mu);
        if (t.enabled && t.calls < kMaxTimedCalls) {
            ev = &t.ev[(size_t)t.calls * (kStages + 1)];
            ++t.calls;
        }
    }
    void mark(int b) {
        if (ev) cudaEventRecord(ev[b], s);
    }
};

int fail(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// ------------------------------------------------------------- pipeline --
// Small-token path (moe_set_small_t_path): 0 = the tcgen05 grouped GEMM for
// every call; 1 = the dequant-GEMV for calls with at most two slots per
// expert on average, when its buffers fit the shared memory at both K (H
// for gate_up, inter for down).
std::atomic<int> g_small_t_path{0};

// Router kernel (moe_set_router_path): 0 = the row router where it fits and
// the clusters would walk two or more waves, 1 = the cluster router always,
// 2 = the row router wherever it fits.
std::atomic<int> g_router_path{0};

bool use_gemv(const moe_dims* d) {
    const long S = (long)d->T * d->k;
    return g_small_t_path.load(std::memory_order_relaxed) == 1 && S <= 2L * d->E && gemv_stages(d->H) >= 2 &&
           gemv_stages(d->inter) >= 2;
}

int run_experts(const moe_dims* d, const uint16_t* x, const int32_t* idx, const uint16_t* w,
                const moe_qweight* gu, const moe_qweight* dn, uint16_t* out, uint8_t* ws, const Layout& L,
                const DeviceInfo& di, cudaStream_t s, CallTimer& tm, const uint16_t* post_norm_w = nullptr) {
    const int S = d->T * d->k;
    const int E = d->E, H = d->H, I = d->inter;
    int32_t* perm = reinterpret_cast<int32_t*>(ws + L.perm);
    int32_t* inv = reinterpret_cast<int32_t*>(ws + L.inv);
    int32_t* offsets = reinterpret_cast<int32_t*>(ws + L.offsets);
    Tile* tiles = reinterpret_cast<Tile*>(ws + L.tiles);
    int32_t* ntiles = reinterpret_cast<int32_t*>(ws + L.ntiles);
    uint16_t* xs = reinterpret_cast<uint16_t*>(ws + L.xs);
    uint16_t* mid = reinterpret_cast<uint16_t*>(ws + L.mid);
    uint16_t* y = reinterpret_cast<uint16_t*>(ws + L.y);
    // A few rows per expert (a decode step): the dequant-GEMV path, which
    // streams the weights without padding the tokens to a tensor-core tile;
    // otherwise the tcgen05 grouped GEMM with token tiles of 64 or 128 rows.
    const bool gemv = use_gemv(d);
    const int nmax = gemv ? kGemvRows : (S / E > 40) ? 128 : 64;

    CUtensorMap m_gu, m_dn;
    BMaps m_xs, m_mid;
    if (!make_map_2d(&m_gu, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, gu->w, H / 8, (uint64_t)E * 2 * I, 32, 64) ||
        !make_map_2d(&m_dn, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, dn->w, I / 8, (uint64_t)E * H, 32, 128) ||
        (!gemv && (!make_bmaps(&m_xs, xs, H, S) || !make_bmaps(&m_mid, mid, I, S))))
        return MOE_ERR_CUDA;

    DispatchArgs da{idx, perm, offsets, inv, tiles, ntiles, S, E, nmax, reinterpret_cast<int32_t*>(ws + L.dhist)};
    int rc;
    if (S <= kDispatchSingleMaxSlots) {  // one launch: every CTA sorts, then gathers its rows
        rc = fail(launch_dispatch_gather(da, x, xs, d->k, H, di.sms, s));
        if (rc) return rc;
        tm.mark(2);
        tm.mark(3);
    } else {
        rc = fail(launch_dispatch(da, s));
        if (rc) return rc;
        tm.mark(2);
        rc = fail(launch_gather(x, perm, offsets, xs, S, d->k, H, E, s));
        if (rc) return rc;
        tm.mark(3);
    }

    GemmArgs ga{};
    ga.scales = gu->scales;
    ga.biases = gu->biases;
    ga.tiles = tiles;
    ga.num_tiles = ntiles;
    ga.out = mid;
    ga.K = H;
    ga.N = 2 * I;
    ga.inter = I;
    ga.out_ld = I;
    ga.nmax = nmax;
    ga.E = E;
    ga.n_tiles = I / 64;
    // With small token tiles the kernels stream weights: warm L2 with each
    // CTA's first two items while the router, dispatch and gather run
    // (guess: token tile t is expert t's, as when every expert has between
    // one and nmax rows). With fewer slots than experts most experts get
    // none and the guess would fetch weights nobody reads: no warm-up.
    ga.w = reinterpret_cast<const uint8_t*>(gu->w);
    ga.prefetch_items = (nmax <= 64 && S >= E) ? 2 : 0;
    ga.tiles_per_expert = 1;
    if (gemv) {
        ga.wstages = gemv_stages(H);
    } else {
        gemm_stages(kGateUp, H, nmax, &ga.wstages, &ga.bregion);
    }
    int grid = di.sms;
    if ((long)L.max_tiles * ga.n_tiles < grid) grid = L.max_tiles * ga.n_tiles;
    rc = fail(gemv ? launch_gemv(kGateUp, m_gu, ga, xs, grid, s) : launch_gemm(kGateUp, m_gu, m_xs, ga, grid, s));
    if (rc) return rc;
    tm.mark(4);

    GemmArgs gd = ga;
    gd.scales = dn->scales;
    gd.biases = dn->biases;
    gd.w = reinterpret_cast<const uint8_t*>(dn->w);
    gd.out = y;
    gd.K = I;
    gd.N = H;
    gd.inter = I;
    gd.out_ld = H;
    gd.n_tiles = H / 128;
    if (gemv) {
        gd.wstages = gemv_stages(I);
    } else {
        gemm_stages(kDown, I, nmax, &gd.wstages, &gd.bregion);
    }
    grid = di.sms;
    if ((long)L.max_tiles * gd.n_tiles < grid) grid = L.max_tiles * gd.n_tiles;
    rc = fail(gemv ? launch_gemv(kDown, m_dn, gd, mid, grid, s) : launch_gemm(kDown, m_dn, m_mid, gd, grid, s));
    if (rc) return rc;
    tm.mark(5);

    rc = fail(post_norm_w ? launch_combine_norm(y, inv, w, post_norm_w, out, d->T, d->k, H, d->eps, s)
                          : launch_combine(y, inv, w, out, d->T, d->k, H, s));
    if (rc) return rc;
    tm.mark(6);
    return MOE_OK;
}

// The dense 4-bit GeGLU MLP on the grouped GEMMs: one expert (E = 1, k = 1)
// whose token tiles cover all T rows. x -> [pre norm] -> gate_up + GeGLU ->
// down -> [post norm, after adding `embeds` when given] -> out.
int run_dense(const moe_dims* d, const uint16_t* x, const uint16_t* pre_norm_w, const uint16_t* embeds,
              const uint16_t* post_norm_w, bool post_norm, const moe_qweight* gu, const moe_qweight* dn, uint16_t* out,
              uint8_t* ws, const Layout& L, const DeviceInfo& di, cudaStream_t s) {
    const int T = d->T, H = d->H, I = d->inter;
    Tile* tiles = reinterpret_cast<Tile*>(ws + L.tiles);
    int32_t* ntiles = reinterpret_cast<int32_t*>(ws + L.ntiles);
    uint16_t* xs = reinterpret_cast<uint16_t*>(ws + L.xs);
    uint16_t* mid = reinterpret_cast<uint16_t*>(ws + L.mid);
    uint16_t* y = reinterpret_cast<uint16_t*>(ws + L.y);
    // 128-row token tiles once they alone give every SM a gate_up item,
    // else 64-row tiles (twice the items, half the MMA width each)
    const int gu_tiles = I / 64;
    const int nmax = ((long)((T + 127) / 128) * gu_tiles >= di.sms) ? 128 : 64;
    const int ntok = (T + nmax - 1) / nmax;

    CUtensorMap m_gu, m_dn;
    BMaps m_xs, m_mid;
    if (!make_map_2d(&m_gu, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, gu->w, H / 8, (uint64_t)2 * I, 32, 64) ||
        !make_map_2d(&m_dn, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, dn->w, I / 8, (uint64_t)H, 32, 128) ||
        !make_bmaps(&m_xs, xs, H, T) || !make_bmaps(&m_mid, mid, I, T))
        return MOE_ERR_CUDA;

    CallTimer tm(s);
    tm.mark(0);
    tm.mark(1);
    tm.mark(2);
    int rc = fail(launch_dense_prep(x, pre_norm_w, d->eps, xs, tiles, ntiles, T, H, nmax, s));
    if (rc) return rc;
    tm.mark(3);

    GemmArgs ga{};
    ga.scales = gu->scales;
    ga.biases = gu->biases;
    ga.tiles = tiles;
    ga.num_tiles = ntiles;
    ga.out = mid;
    ga.K = H;
    ga.N = 2 * I;
    ga.inter = I;
    ga.out_ld = I;
    ga.nmax = nmax;
    ga.E = 1;
    ga.n_tiles = gu_tiles;
    ga.w = reinterpret_cast<const uint8_t*>(gu->w);
    ga.prefetch_items = 2;
    ga.tiles_per_expert = ntok;  // every item is expert 0's
    ga.weight_major = 1;
    gemm_stages(kGateUp, H, nmax, &ga.wstages, &ga.bregion);
    int grid = di.sms < ntok * ga.n_tiles ? di.sms : ntok * ga.n_tiles;
    if ((rc = fail(launch_gemm(kGateUp, m_gu, m_xs, ga, grid, s)))) return rc;
    tm.mark(4);

    GemmArgs gd = ga;
    gd.scales = dn->scales;
    gd.biases = dn->biases;
    gd.w = reinterpret_cast<const uint8_t*>(dn->w);
    gd.out = post_norm ? y : out;
    gd.K = I;
    gd.N = H;
    gd.out_ld = H;
    gd.n_tiles = H / 128;
    gemm_stages(kDown, I, nmax, &gd.wstages, &gd.bregion);
    grid = di.sms < ntok * gd.n_tiles ? di.sms : ntok * gd.n_tiles;
    if ((rc = fail(launch_gemm(kDown, m_dn, m_mid, gd, grid, s)))) return rc;
    tm.mark(5);
    if (post_norm && (rc = fail(launch_add_norm(embeds, y, post_norm_w, d->eps, out, T, H, s)))) return rc;
    tm.mark(6);
    return MOE_OK;
}

// The tied head: h -> interleaved staging -> one-expert GEMM over the vocab
// rows of the 4-bit table with the softcap epilogue (fp32 logits).
int run_head(const moe_dims* d, int vocab, float softcap, const uint16_t* h, const moe_qweight* embed, float* logits,
             uint8_t* ws, const Layout& L, const DeviceInfo& di, cudaStream_t s) {
    const int T = d->T, H = d->H;
    Tile* tiles = reinterpret_cast<Tile*>(ws + L.tiles);
    int32_t* ntiles = reinterpret_cast<int32_t*>(ws + L.ntiles);
    uint16_t* xs = reinterpret_cast<uint16_t*>(ws + L.xs);
    // a vocab-sized weight gives every SM many items: 128-row token tiles
    // (twice the MMA work per dequantised stage) unless T fits one 64-row tile
    const int nmax = T > 64 ? 128 : 64;
    const int ntok = (T + nmax - 1) / nmax;
    const int n_tiles = vocab / 128;

    CUtensorMap m_w;
    BMaps m_xs;
    if (!make_map_2d(&m_w, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, embed->w, H / 8, (uint64_t)vocab, 32, 128) ||
        !make_bmaps(&m_xs, xs, H, T))
        return MOE_ERR_CUDA;
    CallTimer tm(s);
    tm.mark(0);
    tm.mark(1);
    tm.mark(2);
    int rc = fail(launch_dense_prep(h, nullptr, 0.f, xs, tiles, ntiles, T, H, nmax, s));
    if (rc) return rc;
    tm.mark(3);
    GemmArgs ga{};
    ga.scales = embed->scales;
    ga.biases = embed->biases;
    ga.tiles = tiles;
    ga.num_tiles = ntiles;
    ga.out_f32 = logits;
    ga.softcap = softcap;
    ga.K = H;
    ga.N = vocab;
    ga.inter = 0;
    ga.out_ld = vocab;
    ga.nmax = nmax;
    ga.E = 1;
    ga.n_tiles = n_tiles;
    ga.w = reinterpret_cast<const uint8_t*>(embed->w);
    ga.prefetch_items = 2;
    ga.tiles_per_expert = ntok;
    ga.weight_major = 1;
    gemm_stages(kHead, H, nmax, &ga.wstages, &ga.bregion);
    const long items = (long)ntok * n_tiles;
    const int grid = items < di.sms ? (int)items : di.sms;
    if ((rc = fail(launch_gemm(kHead, m_w, m_xs, ga, grid, s)))) return rc;
    tm.mark(4);
    tm.mark(5);
    tm.mark(6);
    return MOE_OK;
}

int check_dense(const moe_dims* d) {
    int rc = check_dims(d);
    if (rc) return rc;
    return (d->E == 1 && d->k == 1) ? MOE_OK : MOE_ERR_SHAPE;
}

int route_impl(const moe_dims* d, const uint16_t* x, const uint16_t* rw, const uint16_t* rs, const uint16_t* pes,
               int32_t* idx, uint16_t* w, cudaStream_t s, const uint16_t* pre_norm_w = nullptr,
               uint16_t* xe = nullptr, const moe_qweight* rq = nullptr) {
    // The row router (one CTA per 16 tokens over the whole row, no cross-CTA
    // exchange) when the cluster router would walk two or more waves of
    // tiles; the cluster router otherwise and for the 4-bit projection.
    const int rpath = g_router_path.load(std::memory_order_relaxed);
    const bool rows = rq == nullptr && ((rpath == 0 && router_prefer_rows(d->T, d->H, d->E)) ||
                                        (rpath == 2 && router_rows_fits(d->H, d->E, false)));
    const int tt = rows ? 16 : router_tokens_per_cluster(d->T, d->H, d->E);
    RouterArgs ra{x,    rw,   rs,   pes,  idx,    w,
                  d->T, d->H, d->E, d->k, d->eps, bf16_round(pow((double)d->H, -0.5)),
                  tt,   pre_norm_w, xe, rq ? rq->w : nullptr, rq ? rq->scales : nullptr,
                  rq ? rq->biases : nullptr};
    CUtensorMap m_rw, m_x;
    if (!make_map_2d(&m_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, d->H, d->T, 64, tt)) return MOE_ERR_CUDA;
    if (rq)
        m_rw = m_x;  // not read: the 4-bit projection is dequantised in the kernel
    else if (!make_map_2d(&m_rw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rw, d->H, d->E, 64, d->E < 128 ? d->E : 128))
        return MOE_ERR_CUDA;
    return fail(rows ? launch_router_rows(m_rw, m_x, ra, s) : launch_router(m_rw, m_x, ra, s));
}

int get_workspace(const moe_dims* d, void* workspace, size_t ws_bytes, const Layout& L, uint8_t** out) {
    if (workspace) {
        if (!aligned16(workspace)) return MOE_ERR_ALIGN;
        if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
        *out = static_cast<uint8_t*>(workspace);
        return MOE_OK;
    }
    void* p = nullptr;
    int rc = owned_workspace(L.total, &p);
    *out = static_cast<uint8_t*>(p);
    return rc;
}

// Scratch of moe_dispatch's large-input path (kDispatchMaxChunks x 256
// ints), allocated once per device on first use and held until the process
// exits.
int dispatch_scratch(int32_t** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_DEVICE;
    static std::mutex mu;
    static std::vector<void*> bufs;
    std::lock_guard<std::mutex> lock(mu);
    if ((int)bufs.size() <= dev) bufs.resize(dev + 1, nullptr);
    if (!bufs[dev] && cudaMalloc(&bufs[dev], (size_t)kDispatchMaxChunks * 256 * 4) != cudaSuccess) {
        bufs[dev] = nullptr;
        return MOE_ERR_CUDA;
    }
    *out = static_cast<int32_t*>(bufs[dev]);
    return MOE_OK;
}

// ------------------------------------------------------ fixed scratch ----
// Scratch of moe_experts_noalloc: a fixed array in the library's device
// image, so that call never allocates. Every GPU that loads the library holds
// it until the process exits. Host code must not use the array's name as a
// device address (on the host it only stands for the symbol); the device
// address comes from cudaGetSymbolAddress, once per device.
constexpr size_t kNoAllocScratchBytes = MOE_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

int noalloc_scratch(uint8_t** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_DEVICE;
    static std::mutex mu;
    static std::vector<void*> ptrs;
    std::lock_guard<std::mutex> lock(mu);
    if ((int)ptrs.size() <= dev) ptrs.resize(dev + 1, nullptr);
    if (!ptrs[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
        ptrs[dev] = p;
    }
    *out = static_cast<uint8_t*>(ptrs[dev]);
    return MOE_OK;
}

}  // namespace

extern "C" {

const char* moe_status_str(int status) {
    switch (status) {
        case MOE_OK: return "ok";
        case MOE_ERR_NULL: return "null pointer";
        case MOE_ERR_SHAPE: return "bad shape";
        case MOE_ERR_ALIGN: return "pointer not 16-byte aligned";
        case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
        case MOE_ERR_WORKSPACE: return "workspace too small";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_TIMEOUT: return "kernel wait timed out";
        case MOE_ERR_DEVICE: return "no usable GPU (needs compute capability 10.3, sm_103a)";
        default: return "unknown status";
    }
}

int moe_workspace_map_of(const moe_dims* d, moe_workspace_map* map) {
    int rc = check_dims(d);
    if (rc) return rc;
    if (!map) return MOE_ERR_NULL;
    const Layout L = layout(d);
    map->idx = L.idx;
    map->w = L.w;
    map->perm = L.perm;
    map->inv = L.inv;
    map->offsets = L.offsets;
    return MOE_OK;
}

size_t moe_workspace_bytes(const moe_dims* d) {
    if (check_dims(d) != MOE_OK) return 0;
    return layout(d).total;
}

int moe_route(const moe_dims* d, const uint16_t* x, const uint16_t* router_w, const uint16_t* router_scale,
              const uint16_t* per_expert_scale, int32_t* idx_out, uint16_t* w_out, void* stream) {
    int rc = check_dims(d);
    if (rc) return rc;
    if ((rc = check_ptrs({x, router_w, router_scale, per_expert_scale, idx_out, w_out}))) return rc;
    if (d->T == 0) return MOE_OK;
    DeviceInfo di;
    if ((rc = device_info(&di))) return rc;
    return route_impl(d, x, router_w, router_scale, per_expert_scale, idx_out, w_out,
                      static_cast<cudaStream_t>(stream));
}

int moe_dispatch(const moe_dims* d, const int32_t* idx, int32_t* perm, int32_t* offsets, int32_t* inv,
                 void* stream) {
    int rc = check_dims(d);
    if (rc) return rc;
    if ((rc = check_ptrs({idx, perm, offsets, inv}))) return rc;
    DeviceInfo di;
    if ((rc = device_info(&di))) return rc;
    int32_t* scratch = nullptr;  // chunk histograms of the large-input path
    if ((rc = dispatch_scratch(&scratch))) return rc;
    DispatchArgs da{idx, perm, offsets, inv, nullptr, nullptr, d->T * d->k, d->E, 64, scratch};
    return fail(launch_dispatch(da, static_cast<cudaStream_t>(stream)));
}

int moe_experts(const moe_dims* d, const uint16_t* x, const int32_t* idx, const uint16_t* w,
                const moe_qweight* gate_up, const moe_qweight* down, uint16_t* out, void* workspace,
                size_t ws_bytes, void* stream) {
    int rc = check_dims(d);
    if (rc) return rc;
    if ((rc = check_ptrs({x, idx, w, out}))) return rc;
    if ((rc = check_qweight(gate_up)) || (rc = check_qweight(down))) return rc;
    if (d->T == 0) return MOE_OK;
    DeviceInfo di;
    if ((rc = device_info(&di))) return rc;
    const Layout L = layout(d);
    uint8_t* ws = nullptr;
    if ((rc = get_workspace(d, workspace, ws_bytes, L, &ws))) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    CallTimer tm(s);
    tm.mark(0);
    tm.mark(1);
    return run_experts(d, x, idx, w, gate_up, down, out, ws, L, di, s, tm);
}

int moe_experts_noalloc(const moe_dims* d, const uint16_t* x, const int32_t* idx, const uint16_t* w,
                        const moe_qweight* gate_up, const moe_qweight* down, uint16_t* out, void* stream) {
    int rc = check_dims(d);
    if (rc) return rc;
    if ((rc = check_ptrs({x, idx, w, out}))) return rc;
    if ((rc = check_qweight(gate_up)) || (rc = check_qweight(down))) return rc;
    const Layout L = layout(d);
    if (L.total > kNoAllocScratchBytes) return MOE_ERR_WORKSPACE;  // beyond the fixed scratch
    if (d->T == 0) return MOE_OK;
    DeviceInfo di;
    if ((rc = device_info(&di))) return rc;
    uint8_t* ws = nullptr;
    if ((rc = noalloc_scratch(&ws))) return rc;
    // Nothing in the scratch has to start at zero: every region the kernels
    // read (routing copy, permutation, offsets, tile list, gathered inputs,
    // GeGLU output, expert outputs) is written earlier in the same call.
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    CallTimer tm(s);
    tm.mark(0);
    tm.mark(1);
    return run_experts(d, x, idx, w, gate_up, down, out, ws, L, di, s, tm);
}

int moe_forward(const moe_dims* d, const uint16_t* x, const uint16_t* router_w, const uint16_t* router_scale,
                const uint16_t* per_expert_scale, const moe_qweight* gate_up, const moe_qweight* down,
                uint16_t* out, int32_t* idx_out, uint16_t* w_out, void* workspace, size_t ws_bytes,
                void* stream) {
    int rc = check_dims(d);
    if (rc) return rc;
    if ((rc = check_ptrs({x, router_w, router_scale, per_expert_scale, out}))) return rc;
    if ((rc = check_qweight(gate_up)) || (rc = check_qweight(down))) return rc;
    if ((idx_out && !aligned16(idx_out)) || (w_out && !aligned16(w_out))) return MOE_ERR_ALIGN;
    if (d->T == 0) return MOE_OK;
    DeviceInfo di;
    if ((rc = device_info(&di))) return rc;
    const Layout L = layout(d);
    uint8_t* ws = nullptr;
    if ((rc = get_workspace(d, workspace, ws_bytes, L, &ws))) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t* idx = idx_out ? idx_out : reinterpret_cast<int32_t*>(ws + L.idx);
    uint16_t* w = w_out ? w_out : reinterpret_cast<uint16_t*>(ws + L.w);
    CallTimer tm(s);
    tm.mark(0);
    if ((rc = route_impl(d, x, router_w, router_scale, per_expert_scale, idx, w, s))) return rc;
    tm.mark(1);
    return run_experts(d, x, idx, w, gate_up, down, out, ws, L, di, s, tm);
}

int moe_route_q4(const moe_dims* d, const uint16_t* x, const moe_qweight* router_q, const uint16_t* router_scale,
                 const uint16_t* per_expert_scale, int32_t* idx_out, uint16_t* w_out, void* stream) {
    int rc = check_dims(d);
    if (rc) return rc;
    if ((rc = check_ptrs({x, router_scale, per_expert_scale, idx_out, w_out}))) return rc;
    if ((rc = check_qweight(router_q))) return rc;
    if (d->E > 128) return MOE_ERR_UNSUPPORTED;  // one dequantised chunk of experts
    if (d->T == 0) return MOE_OK;
    return route_impl(d, x, nullptr, router_scale, per_expert_scale, idx_out, w_out, static_cast<cudaStream_t>(stream),
                      nullptr, nullptr, router_q);
}

int moe_forward_q4router(const moe_dims* d, const uint16_t* x, const moe_qweight* router_q,
                         const uint16_t* router_scale, const uint16_t* per_expert_scale, const moe_qweight* gate_up,
                         const moe_qweight* down, uint16_t* out, int32_t* idx_out, uint16_t* w_out, void* workspace,
                         size_t ws_bytes, void* stream) {
    int rc = check_dims(d);
    if (rc) return rc;
    if ((rc = check_ptrs({x, router_scale, per_expert_scale, out}))) return rc;
    if ((rc = check_qweight(router_q)) || (rc = check_qweight(gate_up)) || (rc = check_qweight(down))) return rc;
    if ((idx_out && !aligned16(idx_out)) || (w_out && !aligned16(w_out))) return MOE_ERR_ALIGN;
    if (d->E > 128) return MOE_ERR_UNSUPPORTED;
    if (d->T == 0) return MOE_OK;
    DeviceInfo di;
    if ((rc = device_info(&di))) return rc;
    const Layout L = layout(d);
    uint8_t* ws = nullptr;
    if ((rc = get_workspace(d, workspace, ws_bytes, L, &ws))) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t* idx = idx_out ? idx_out : reinterpret_cast<int32_t*>(ws + L.idx);
    uint16_t* w = w_out ? w_out : reinterpret_cast<uint16_t*>(ws + L.w);
    CallTimer tm(s);
    tm.mark(0);
    if ((rc = route_impl(d, x, nullptr, router_scale, per_expert_scale, idx, w, s, nullptr, nullptr, router_q)))
        return rc;
    tm.mark(1);
    return run_experts(d, x, idx, w, gate_up, down, out, ws, L, di, s, tm);
}

int moe_forward_branch(const moe_dims* d, const uint16_t* residual, const uint16_t* router_w,
                       const uint16_t* router_scale, const uint16_t* per_expert_scale, const uint16_t* pre_norm_w,
                       const uint16_t* post_norm_w, const moe_qweight* gate_up, const moe_qweight* down,
                       uint16_t* out, int32_t* idx_out, uint16_t* w_out, uint16_t* expert_in_out, void* workspace,
                       size_t ws_bytes, void* stream) {
    int rc = check_dims(d);
    if (rc) return rc;
    if ((rc = check_ptrs({residual, router_w, router_scale, per_expert_scale, pre_norm_w, post_norm_w, out})))
        return rc;
    if ((rc = check_qweight(gate_up)) || (rc = check_qweight(down))) return rc;
    if ((idx_out && !aligned16(idx_out)) || (w_out && !aligned16(w_out)) ||
        (expert_in_out && !aligned16(expert_in_out)))
        return MOE_ERR_ALIGN;
    if (d->H > 8192) return MOE_ERR_UNSUPPORTED;  // the post norm's one-CTA-a-token row
    if (d->T == 0) return MOE_OK;
    DeviceInfo di;
    if ((rc = device_info(&di))) return rc;
    const Layout L = layout(d);
    uint8_t* ws = nullptr;
    if ((rc = get_workspace(d, workspace, ws_bytes, L, &ws))) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t* idx = idx_out ? idx_out : reinterpret_cast<int32_t*>(ws + L.idx);
    uint16_t* w = w_out ? w_out : reinterpret_cast<uint16_t*>(ws + L.w);
    uint16_t* xe = expert_in_out ? expert_in_out : reinterpret_cast<uint16_t*>(ws + L.xdev);
    CallTimer tm(s);
    tm.mark(0);
    if ((rc = route_impl(d, residual, router_w, router_scale, per_expert_scale, idx, w, s, pre_norm_w, xe)))
        return rc;
    tm.mark(1);
    return run_experts(d, xe, idx, w, gate_up, down, out, ws, L, di, s, tm, post_norm_w);
}

int moe_dense_mlp(const moe_dims* d, const uint16_t* x, const moe_qweight* gate_up, const moe_qweight* down,
                  uint16_t* out, void* workspace, size_t ws_bytes, void* stream) {
    int rc = check_dense(d);
    if (rc) return rc;
    if ((rc = check_ptrs({x, out}))) return rc;
    if ((rc = check_qweight(gate_up)) || (rc = check_qweight(down))) return rc;
    if (d->T == 0) return MOE_OK;
    DeviceInfo di;
    if ((rc = device_info(&di))) return rc;
    const Layout L = layout(d);
    uint8_t* ws = nullptr;
    if ((rc = get_workspace(d, workspace, ws_bytes, L, &ws))) return rc;
    return run_dense(d, x, nullptr, nullptr, nullptr, false, gate_up, down, out, ws, L, di,
                     static_cast<cudaStream_t>(stream));
}

int moe_dense_branch(const moe_dims* d, const uint16_t* h, const uint16_t* pre_norm_w, const uint16_t* post_norm_w,
                     const moe_qweight* gate_up, const moe_qweight* down, uint16_t* out, void* workspace,
                     size_t ws_bytes, void* stream) {
    int rc = check_dense(d);
    if (rc) return rc;
    if ((rc = check_ptrs({h, pre_norm_w, post_norm_w, out}))) return rc;
    if ((rc = check_qweight(gate_up)) || (rc = check_qweight(down))) return rc;
    if (d->T == 0) return MOE_OK;
    DeviceInfo di;
    if ((rc = device_info(&di))) return rc;
    const Layout L = layout(d);
    uint8_t* ws = nullptr;
    if ((rc = get_workspace(d, workspace, ws_bytes, L, &ws))) return rc;
    return run_dense(d, h, pre_norm_w, nullptr, post_norm_w, true, gate_up, down, out, ws, L, di,
                     static_cast<cudaStream_t>(stream));
}

int moe_self_conditioning(const moe_dims* d, const uint16_t* inputs_embeds, const uint16_t* signal,
                          const uint16_t* pre_norm_w, const moe_qweight* gate_up, const moe_qweight* down,
                          uint16_t* out, void* workspace, size_t ws_bytes, void* stream) {
    int rc = check_dense(d);
    if (rc) return rc;
    if ((rc = check_ptrs({inputs_embeds, signal, pre_norm_w, out}))) return rc;
    if ((rc = check_qweight(gate_up)) || (rc = check_qweight(down))) return rc;
    if (d->T == 0) return MOE_OK;
    DeviceInfo di;
    if ((rc = device_info(&di))) return rc;
    const Layout L = layout(d);
    uint8_t* ws = nullptr;
    if ((rc = get_workspace(d, workspace, ws_bytes, L, &ws))) return rc;
    return run_dense(d, signal, pre_norm_w, inputs_embeds, nullptr, true, gate_up, down, out, ws, L, di,
                     static_cast<cudaStream_t>(stream));
}

int moe_lm_head(const moe_dims* d, int32_t vocab, float softcap, const uint16_t* h, const moe_qweight* embed,
                float* logits, void* workspace, size_t ws_bytes, void* stream) {
    int rc = check_dense(d);
    if (rc) return rc;
    if (vocab <= 0) return MOE_ERR_SHAPE;
    if (vocab % 128 != 0) return MOE_ERR_UNSUPPORTED;  // 128-row weight tiles
    if (!(softcap >= 0.0f) || isinf(softcap)) return MOE_ERR_SHAPE;
    if ((rc = check_ptrs({h, logits}))) return rc;
    if ((rc = check_qweight(embed))) return rc;
    if (d->T == 0) return MOE_OK;
    DeviceInfo di;
    if ((rc = device_info(&di))) return rc;
    const Layout L = layout(d);
    uint8_t* ws = nullptr;
    if ((rc = get_workspace(d, workspace, ws_bytes, L, &ws))) return rc;
    return run_head(d, vocab, softcap, h, embed, logits, ws, L, di, static_cast<cudaStream_t>(stream));
}

int moe_forward_hostio(const moe_dims* d, const uint16_t* x_host, const uint16_t* router_w,
                       const uint16_t* router_scale, const uint16_t* per_expert_scale, const moe_qweight* gate_up,
                       const moe_qweight* down, uint16_t* out_host, void* workspace, size_t ws_bytes,
                       void* stream) {
    int rc = check_dims(d);
    if (rc) return rc;
    if (!x_host || !out_host) return MOE_ERR_NULL;
    if ((rc = check_ptrs({router_w, router_scale, per_expert_scale}))) return rc;
    if ((rc = check_qweight(gate_up)) || (rc = check_qweight(down))) return rc;
    if (d->T == 0) return MOE_OK;
    DeviceInfo di;
    if ((rc = device_info(&di))) return rc;
    const Layout L = layout(d);
    uint8_t* ws = nullptr;
    if ((rc = get_workspace(d, workspace, ws_bytes, L, &ws))) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint16_t* xdev = reinterpret_cast<uint16_t*>(ws + L.xdev);
    uint16_t* odev = reinterpret_cast<uint16_t*>(ws + L.outdev);
    const size_t bytes = (size_t)d->T * d->H * 2;
    // Pinned buffers are mapped into the device's address space: x is read
    // by a copy kernel on every SM and the combine writes out straight into
    // out_host (each over the host link, no copy-engine transfer: 1.44 MB
    // each way took ~27 us through the copy engines at T = 256). Buffers the
    // runtime cannot map (pageable) go through cudaMemcpyAsync.
    void* x_map = nullptr;
    void* o_map = nullptr;
    const bool zx = cudaHostGetDevicePointer(&x_map, const_cast<uint16_t*>(x_host), 0) == cudaSuccess &&
                    aligned16(x_map);
    cudaGetLastError();  // a pageable buffer leaves a (non-sticky) error behind
    const bool zo = cudaHostGetDevicePointer(&o_map, out_host, 0) == cudaSuccess && aligned16(o_map);
    cudaGetLastError();
    if (zx) {
        if ((rc = fail(launch_copy16(xdev, x_map, bytes, di.sms, s)))) return rc;
    } else if (cudaMemcpyAsync(xdev, x_host, bytes, cudaMemcpyHostToDevice, s) != cudaSuccess) {
        return MOE_ERR_CUDA;
    }
    uint16_t* out_dst = zo ? static_cast<uint16_t*>(o_map) : odev;
    rc = moe_forward(d, xdev, router_w, router_scale, per_expert_scale, gate_up, down, out_dst, nullptr, nullptr, ws,
                     L.total, stream);
    if (rc) return rc;
    if (!zo && cudaMemcpyAsync(out_host, odev, bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess) return MOE_ERR_CUDA;
    return fail(cudaStreamSynchronize(s));
}

int moe_set_router_path(int mode) {
    if (mode < 0 || mode > 2) return -MOE_ERR_SHAPE;
    return g_router_path.exchange(mode);
}

int moe_set_small_t_path(int mode) {
    if (mode != 0 && mode != 1) return -MOE_ERR_SHAPE;
    return g_small_t_path.exchange(mode);
}

int moe_timing_enable(int enable) {
    Timing& t = timing();
    std::lock_guard<std::mutex> lock(t.mu);
    if (enable && t.ev.empty()) {
        t.ev.resize((size_t)kMaxTimedCalls * (kStages + 1));
        for (auto& e : t.ev)
            if (cudaEventCreate(&e) != cudaSuccess) return MOE_ERR_CUDA;
    }
    t.enabled = enable != 0;
    t.calls = 0;
    return MOE_OK;
}

int moe_timing_read(float* ms, int n, int* calls) {
    Timing& t = timing();
    std::lock_guard<std::mutex> lock(t.mu);
    const int m = n < kStages ? n : kStages;
    for (int i = 0; i < m; ++i) ms[i] = 0.f;
    for (int c = 0; c < t.calls; ++c) {
        cudaEvent_t* ev = &t.ev[(size_t)c * (kStages + 1)];
        if (cudaEventSynchronize(ev[kStages]) != cudaSuccess) return -MOE_ERR_CUDA;
        for (int i = 0; i < m; ++i) {
            float v = 0.f;
            if (cudaEventElapsedTime(&v, ev[i], ev[i + 1]) == cudaSuccess) ms[i] += v;
        }
    }
    if (calls) *calls = t.calls;
    t.calls = 0;
    return m;
}

int moe_launches_per_forward(const moe_dims* d) {
    if (check_dims(d) != MOE_OK) return 0;
    // router, dispatch fused with the gather, gate_up, down, combine; above
    // 8192 slots the dispatch runs as three kernels and the gather as its own
    return ((int64_t)d->T * d->k > kDispatchSingleMaxSlots) ? 8 : 5;
}

int moe_device_error(void) {
    if (cudaDeviceSynchronize() != cudaSuccess) return -MOE_ERR_CUDA;
    return router_error_word() | dispatch_error_word() | gemm_error_word() | gemv_error_word();
}

}  // extern "C"
