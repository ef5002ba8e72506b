// Router kernel: DiffRouter.forward of the DiffusionGemma language model
// ("diffusion-gemma/model.ts"), fused into one launch.
//
// Thread-block clusters of 8 CTAs, persistent: as many as the device holds at
// once (at most one per tile), each walking token tiles of TT tokens (TT =
// 16, 32 or 64). The hidden dimension is split into 64-wide blocks shared out
// over the cluster: CTA r loads once, by TMA with the 128-byte swizzle, its
// blocks of every router-weight row (kept for all tiles when E <= 128), and
// per tile its blocks of the TT activation rows. Per tile
//   1. each CTA sums the squares of its slice per token (fp32 with an
//      error-free two-sum, so the partial sum keeps ~48 bits) and sends the
//      partial to every CTA of the cluster (distributed shared memory);
//   2. every CTA adds the 8 partials in CTA order, forms the fp32 mean as the
//      two-float sum divided by H and rounded once (the fp32 RMS-norm
//      semantics "diffusion-gemma/vision.ts" spells out in manualRms), and normalises
//      its slice in place, then the two bf16 multiplies (router scale,
//      H^-0.5), bf16 after each op;
//   3. each CTA computes partial scores of all TT tokens x E experts over its
//      slice on the tensor cores (tcgen05.mma, 128 experts on the TMEM lanes,
//      fp32 accumulate) and sends each token's partials to the CTA that owns
//      the token (TT/8 tokens per CTA);
//   4. the owner adds the 8 partials in CTA order, rounds to bf16, picks the
//      top k (value descending, ties to the lower expert id), takes the fp32
//      softmax over the k picked scores and multiplies by
//      per_expert_scale[idx].
// Every CTA passes the same cluster barriers (one at the start, two a tile)
// whatever happens, so a wait that times out (error word set) cannot leave the
// cluster hung. The next tile's activations load during step 4.
#include <cooperative_groups.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <utility>

#include "common.cuh"
#include "kernels.h"

namespace cg = cooperative_groups;

namespace moe {

namespace {

constexpr int kCS = 8;          // CTAs per cluster
constexpr int kWarps = 16;      // warps per CTA
constexpr int kChunkE = 128;    // experts per router-weight chunk in shared memory
constexpr int kWBlockBytes = kChunkE * 128;  // one 64-wide K block of a chunk
constexpr uint32_t kTmemCols = 64;           // >= the largest TT
constexpr int kMaxRouterE = 256;             // top-k candidates: 8 per lane

// bf16 bits -> key that orders like the value (for finite values).
__device__ __forceinline__ uint32_t order_key16(uint32_t b) { return (b & 0x8000u) ? (~b & 0xFFFFu) : (b | 0x8000u); }
__device__ __forceinline__ uint32_t key16_to_bits(uint32_t k) { return (k & 0x8000u) ? (k & 0x7FFFu) : (~k & 0xFFFFu); }

// Byte offset of 16-byte chunk c (0..7) of row r inside a 128-byte-swizzled
// box of 128-byte rows.
__device__ __forceinline__ int sw128(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

// Error-free transformation of a + b (Knuth's two-sum): s + e == a + b exactly.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    const float bp = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp));
}

// (hi, lo) += v, keeping hi + lo within ~2^-48 of the exact running sum.
__device__ __forceinline__ void acc2(float& hi, float& lo, float v) {
    float s, e;
    two_sum(hi, v, s, e);
    hi = s;
    lo = __fadd_rn(lo, e);
}

// K blocks [kb0, kb0 + cnt) of the H / 64 blocks owned by cluster rank r.
__host__ __device__ inline void kslice(int nkb, int r, int& kb0, int& cnt) {
    const int base = nkb / kCS, rem = nkb % kCS;
    cnt = base + (r < rem ? 1 : 0);
    kb0 = r * base + (r < rem ? r : rem);
}

struct RouterSmem {
    uint8_t *xt, *wt, *rsl;  // x slice boxes, weight-chunk blocks, router_scale slice
    uint8_t* psl;            // expert-input norm weight slice (optional output xe)
    float2* pss;             // [kCS][TT] partial sums of squares, by source CTA
    float* red;              // [kCS][TT/kCS][E] partial scores of my tokens, by source CTA
    uint16_t* sc;            // [TT/kCS][E] bf16 scores of my tokens
};

__host__ __device__ inline size_t take_bytes(size_t& off, size_t bytes, size_t align) {
    off = (off + align - 1) & ~(align - 1);
    const size_t at = off;
    off += bytes;
    return at;
}

// Carve-up of the dynamic shared memory (from a 1024-byte aligned base);
// returns its size.
__host__ __device__ inline size_t router_layout(int H, int E, int TT, uint8_t* base, RouterSmem* s) {
    const int nkbmax = (H / 64 + kCS - 1) / kCS;
    size_t off = 0;
    const size_t xt = take_bytes(off, (size_t)nkbmax * TT * 128, 1024);
    const size_t wt = take_bytes(off, (size_t)nkbmax * kWBlockBytes, 1024);
    const size_t rsl = take_bytes(off, (size_t)nkbmax * 128, 16);
    const size_t psl = take_bytes(off, (size_t)nkbmax * 128, 16);
    const size_t pss = take_bytes(off, (size_t)kCS * TT * sizeof(float2), 16);
    const size_t red = take_bytes(off, (size_t)TT * E * sizeof(float), 16);
    const size_t sc = take_bytes(off, (size_t)(TT / kCS) * E * 2, 16);
    if (s) {
        s->xt = base + xt;
        s->wt = base + wt;
        s->rsl = base + rsl;
        s->psl = base + psl;
        s->pss = reinterpret_cast<float2*>(base + pss);
        s->red = reinterpret_cast<float*>(base + red);
        s->sc = reinterpret_cast<uint16_t*>(base + sc);
    }
    return off;
}

}  // namespace

__global__ void __launch_bounds__(kWarps * 32) router_kernel(const __grid_constant__ CUtensorMap wmap,
                                                              const __grid_constant__ CUtensorMap xmap,
                                                              RouterArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ uint64_t full, wfull, mdone;
    __shared__ uint32_t tmem_base;
    __shared__ uint16_t pes_s[kMaxRouterE];  // per_expert_scale
    __shared__ float rs_s[64];               // 1 / rms of each token of the tile
    __shared__ int abort_flag_s;
    pdl_trigger();
    pdl_wait();
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int H = a.H, E = a.E, k = a.k, TT = a.tt;
    RouterSmem sm;
    router_layout(H, E, TT, base, &sm);
    volatile int* abort_flag = &abort_flag_s;

    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int cl = (int)blockIdx.x / kCS, ncl = (int)gridDim.x / kCS;  // this cluster, clusters
    const int ntiles = (a.T + TT - 1) / TT;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int kb0, cnt;
    kslice(H / 64, rank, kb0, cnt);
    const int nch = (E + kChunkE - 1) / kChunkE;
    const int eb = E < kChunkE ? E : kChunkE;  // rows of a weight box
    const int tpc = TT / kCS;                  // tokens owned by each CTA

    for (int e = threadIdx.x; e < E; e += blockDim.x) pes_s[e] = a.per_expert_scale[e];
    const bool wq = a.rq_w != nullptr;  // 4-bit projection, dequantised below
    if (threadIdx.x == 0) {
        prefetch_tensormap(&xmap);
        if (!wq) prefetch_tensormap(&wmap);
        mbar_init(&full, 1);
        mbar_init(&wfull, 1);
        mbar_init(&mdone, 1);
        abort_flag_s = 0;
        fence_barrier_init();
    }
    __syncthreads();
    // Copies of tile `tile`'s activation slice (and, with `weights`, of the
    // first weight chunk and the router scale slice), one lane per copy. They
    // only write this CTA's shared memory.
    auto issue_loads = [&](int tile, bool weights) {
        if (lane == 0)
            mbar_arrive_expect_tx(&full, (uint32_t)cnt * (TT * 128 + (weights ? (wq ? 0 : eb * 128) + 128 : 0) +
                                                          (weights && a.xe ? 128 : 0)));
        __syncwarp();
        if (lane < cnt) tma_load_2d(sm.xt + lane * TT * 128, &xmap, &full, (kb0 + lane) * 64, tile * TT);
        if (weights && !wq && lane >= 16 && lane - 16 < cnt)
            tma_load_2d(sm.wt + (lane - 16) * kWBlockBytes, &wmap, &full, (kb0 + lane - 16) * 64, 0);
        if (weights && lane == 31 && cnt > 0) bulk_load(sm.rsl, a.router_scale + (size_t)kb0 * 64, cnt * 128, &full);
        if (weights && a.xe && lane == 30 && cnt > 0) bulk_load(sm.psl, a.pre_w + (size_t)kb0 * 64, cnt * 128, &full);
    };
    if (warp == 0) {  // scores accumulator: 128 lanes (experts) x TT columns (tokens)
        tmem_alloc(&tmem_base, kTmemCols);
        tmem_relinquish();
    } else if (warp == 1 && cl < ntiles) {
        issue_loads(cl, true);
    }
    // Cluster barrier 0: every CTA's barriers exist before any remote write.
    tc_fence_before();
    cluster_barrier();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    if (wq) {
        // This CTA's blocks of the 4-bit projection, once: word j of row e in
        // block kb holds elements 8j..8j+7 of that block (low nibble first),
        // i.e. 16-byte chunk j of the row, stored at chunk j ^ (e % 8) as the
        // 128-byte swizzle of the copies lays it out. w = bf16(S q + B): the
        // product of a bf16 scale and a 4-bit code is exact, the sum rounds
        // once to fp32 and once to bf16 (exact in fp32 for these operands).
        const int G = H / 64, W8 = H / 8;
        for (int i = threadIdx.x; i < E * cnt * 8; i += kWarps * 32) {
            const int j = i & 7, kb = (i >> 3) % cnt, e = (i >> 3) / cnt;
            const uint32_t word = __ldg(a.rq_w + (size_t)e * W8 + (size_t)(kb0 + kb) * 8 + j);
            const float S = bf16_bits_to_f32(__ldg(a.rq_s + (size_t)e * G + kb0 + kb));
            const float B = bf16_bits_to_f32(__ldg(a.rq_b + (size_t)e * G + kb0 + kb));
            uint32_t v[4];
#pragma unroll
            for (int p = 0; p < 4; ++p)
                v[p] = pack_bf16x2(__fmaf_rn(S, (float)((word >> (8 * p)) & 0xFu), B),
                                   __fmaf_rn(S, (float)((word >> (8 * p + 4)) & 0xFu), B));
            *reinterpret_cast<uint4*>(sm.wt + kb * kWBlockBytes + e * 128 + ((j ^ (e & 7)) << 4)) =
                make_uint4(v[0], v[1], v[2], v[3]);
        }
        // visible to the MMAs (async proxy) after phase 2's proxy fence and barrier
    }
    const uint32_t rootb = f32_to_bf16_bits(a.root), root2 = rootb | (rootb << 16);
    uint32_t ncommit = 0, nreload = 0;  // mdone and wfull phases used so far

    // Persistent over token tiles: the cluster keeps its weight slice in
    // shared memory (one chunk when E <= 128) and walks tiles cl, cl + ncl,
    // ... Per tile two cluster barriers; the next tile's activations load
    // while this tile's top k runs. Every CTA of the cluster walks the same
    // tiles and passes the same barriers whatever happens.
    int it = 0;
    for (int tile = cl; tile < ntiles; tile += ncl, ++it) {
        const int t0 = tile * TT;
        const bool have = mbar_wait(&full, (uint32_t)it & 1, abort_flag);

        // ---- 1. partial sums of squares of this slice, to every CTA ----
        // 512 / TT threads a token (8, 16 or 32 adjacent lanes of a warp),
        // thread `sub` summing chunks sub, sub + tpt, ... of the token's
        // slice in two independent two-float accumulators (alternate chunks),
        // so no thread runs one long dependent chain. The merge and the
        // butterfly over the token's threads are error-free two-sums, whose
        // results do not depend on operand order, so every thread of the
        // token ends with the same value.
        {
            const int tpt = (kWarps * 32) / TT;
            const int t = (int)threadIdx.x / tpt, sub = (int)threadIdx.x % tpt;
            const int nchunk = have ? cnt * 8 : 0;
            float h0 = 0.f, l0 = 0.f, h1 = 0.f, l1 = 0.f;
            for (int i = sub; i < nchunk; i += 2 * tpt) {
                const uint4 v = *reinterpret_cast<const uint4*>(sm.xt + (i >> 3) * TT * 128 + sw128(t, i & 7));
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                const int i2 = i + tpt;
                uint4 v2 = make_uint4(0u, 0u, 0u, 0u);
                if (i2 < nchunk) v2 = *reinterpret_cast<const uint4*>(sm.xt + (i2 >> 3) * TT * 128 + sw128(t, i2 & 7));
                const uint32_t w2[4] = {v2.x, v2.y, v2.z, v2.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    // squares of bf16 values are exact in fp32 (zero chunks add nothing)
                    const float x0 = bf16_bits_to_f32(w[j] & 0xFFFFu), x1 = bf16_bits_to_f32(w[j] >> 16);
                    const float y0 = bf16_bits_to_f32(w2[j] & 0xFFFFu), y1 = bf16_bits_to_f32(w2[j] >> 16);
                    acc2(h0, l0, __fmul_rn(x0, x0));
                    acc2(h1, l1, __fmul_rn(y0, y0));
                    acc2(h0, l0, __fmul_rn(x1, x1));
                    acc2(h1, l1, __fmul_rn(y1, y1));
                }
            }
            float hi, lo, se;
            two_sum(h0, h1, hi, se);
            lo = __fadd_rn(__fadd_rn(l0, l1), se);
            for (int o = tpt / 2; o > 0; o >>= 1) {
                const float h2 = __shfl_xor_sync(0xffffffffu, hi, o), l2 = __shfl_xor_sync(0xffffffffu, lo, o);
                float s2, e2;
                two_sum(hi, h2, s2, e2);
                hi = s2;
                lo = __fadd_rn(__fadd_rn(lo, l2), e2);
            }
            if (sub < kCS) cluster.map_shared_rank(sm.pss, sub)[rank * TT + t] = make_float2(hi, lo);
        }
        __syncwarp();
        cluster_barrier();  // A: all partial sums of squares delivered

        // ---- 2. rsqrt of the fp32 mean (a thread a token), normalise this slice in place ----
        if ((int)threadIdx.x < TT) {
            const int t = threadIdx.x;
            float hs = 0.f, ls = 0.f;
            for (int src = 0; src < kCS; ++src) {  // CTA order: the same result in every CTA
                const float2 p = sm.pss[src * TT + t];
                acc2(hs, ls, p.x);
                ls = __fadd_rn(ls, p.y);
            }
            // mean = (hs + ls) / H rounded once to fp32, without fp64 (slow on
            // this part): q = RN(hs / H); the residual hs - q H is exact
            // (fma); adding (residual + ls) / H moves q by under half an ulp,
            // so the sum rounds to the exactly rounded mean unless that mean
            // lies within about 2^-40 (relative) of a rounding boundary.
            const float Hf = (float)H;
            const float q0 = __fdiv_rn(hs, Hf);
            const float rsd = __fadd_rn(__fmaf_rn(-q0, Hf, hs), ls);
            const float mean = __fadd_rn(q0, __fdiv_rn(rsd, Hf));
            rs_s[t] = __frsqrt_rn(__fadd_rn(mean, a.eps));
        }
        __syncthreads();
        // bf16 after each op: x*rs in fp32 rounded once (cvt.rn), then the
        // two bf16 x bf16 products, each exact in fp32 and rounded once
        // (mul.rn.bf16x2), two elements an instruction. Element i of the
        // loop is token i % TT, chunk i / TT of the slice.
        {
            const int nchunk = cnt * 8;
            const int tshift = 31 - __clz(TT);
            for (int i = threadIdx.x; have && i < TT * nchunk; i += kWarps * 32) {
                const int t = i & (TT - 1), c = i >> tshift;
                const float rs = rs_s[t];
                uint4* p = reinterpret_cast<uint4*>(sm.xt + (c >> 3) * TT * 128 + sw128(t, c & 7));
                const uint4 v = *p;
                if (a.xe && t0 + t < a.T) {  // the expert input: bf16((x * rs) * pre_w), one rounding
                    const uint4 pw = reinterpret_cast<const uint4*>(sm.psl)[c];
                    const uint32_t xv[4] = {v.x, v.y, v.z, v.w}, wv[4] = {pw.x, pw.y, pw.z, pw.w};
                    uint32_t e[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        e[j] = pack_bf16x2(
                            __fmul_rn(__fmul_rn(__uint_as_float(xv[j] << 16), rs), __uint_as_float(wv[j] << 16)),
                            __fmul_rn(__fmul_rn(__uint_as_float(xv[j] & 0xFFFF0000u), rs),
                                      __uint_as_float(wv[j] & 0xFFFF0000u)));
                    const size_t h = (size_t)(kb0 + (c >> 3)) * 64 + (c & 7) * 8;
                    *reinterpret_cast<uint4*>(a.xe + (size_t)(t0 + t) * H + h) = make_uint4(e[0], e[1], e[2], e[3]);
                }
                const uint4 sv = reinterpret_cast<const uint4*>(sm.rsl)[c];  // router_scale of the same 8 columns
                const uint32_t w[4] = {v.x, v.y, v.z, v.w}, sc[4] = {sv.x, sv.y, sv.z, sv.w};
                uint32_t o[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t n = pack_bf16x2(__fmul_rn(__uint_as_float(w[j] << 16), rs),
                                                   __fmul_rn(__uint_as_float(w[j] & 0xFFFF0000u), rs));
                    o[j] = mul_bf16x2(mul_bf16x2(n, sc[j]), root2);
                }
                *p = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
        // The normalised tile was written by ordinary stores; the tensor core
        // reads it through the async proxy.
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();

        // ---- 3. partial scores over this slice, to the CTA owning each token ----
        // D[e][t] = sum over this slice of W[e][h] * n[t][h], experts on the
        // 128 TMEM lanes and tokens on TT columns: one tcgen05.mma per 16 K
        // (A = the weight chunk, B = the normalised tile, both K-major in
        // shared memory).
        const uint32_t idesc = idesc_bf16_m128((uint32_t)TT);
        for (int ch = 0; ch < nch; ++ch) {
            bool wok = have;
            // With more than one chunk, chunk ch (and chunk 0 again from the
            // second tile on) is reloaded into the weight buffer.
            if (ch > 0 || (nch > 1 && it > 0)) {
                __syncthreads();  // every warp has read the previous chunk's scores
                if (threadIdx.x == 0) {
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    mbar_arrive_expect_tx(&wfull, (uint32_t)cnt * eb * 128);
                    for (int i = 0; i < cnt; ++i)
                        tma_load_2d(sm.wt + i * kWBlockBytes, &wmap, &wfull, (kb0 + i) * 64, ch * kChunkE);
                }
                wok = mbar_wait(&wfull, nreload & 1, abort_flag) && wok;
                ++nreload;
            }
            const bool mma = wok && cnt > 0;
            if (warp == 0 && mma) {
                tc_fence_after();
                if (elect_one()) {
                    for (int kb = 0; kb < cnt; ++kb) {
                        const uint64_t ad = sw128_kmajor_desc(smem_u32(sm.wt + kb * kWBlockBytes));
                        const uint64_t bd = sw128_kmajor_desc(smem_u32(sm.xt + kb * TT * 128));
#pragma unroll
                        for (int k16 = 0; k16 < 4; ++k16)
                            umma_ss(tmem, ad + (uint64_t)(k16 * 2), bd + (uint64_t)(k16 * 2), idesc,
                                    (kb > 0 || k16 > 0) ? 1u : 0u);
                    }
                    umma_commit(&mdone);
                }
                __syncwarp();
            }
            // Every CTA of the cluster commits (or skips) the same MMAs, so
            // the phase count stays in step; a skipped commit leaves the
            // count unchanged.
            const bool got = mma && mbar_wait(&mdone, ncommit & 1, abort_flag);
            if (mma) ++ncommit;
            tc_fence_after();
            // Warp w reads TMEM lane quarter w % 4 (experts ch*128 + 32(w%4) +
            // lane) and the 16 token columns 16 (w / 4) .. 16 (w / 4) + 15.
            const int e = ch * kChunkE + (warp & 3) * 32 + lane;
            const int c0 = (warp >> 2) * 16;
            if (c0 < TT) {
                uint32_t v[16];
                if (got) {
                    tmem_ld16(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)c0, v);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[j] = 0u;  // no K blocks here (or a wait timed out)
                }
                if (e < E) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int tok = c0 + j;
                        cluster.map_shared_rank(sm.red, tok / tpc)[(size_t)(rank * tpc + tok % tpc) * E + e] =
                            __uint_as_float(v[j]);
                    }
                }
            }
            tc_fence_before();
        }
        __syncwarp();
        cluster_barrier();  // B: all partial scores delivered; no remote access until A of the next tile

        // The activation buffer is free (the MMAs read it before their
        // commit): load the next tile's slice while this tile's top k runs.
        if (warp == 1 && tile + ncl < ntiles) issue_loads(tile + ncl, false);

        // ---- 4. my tokens: scores, top k, precise softmax, per-expert scale ----
        for (int i = threadIdx.x; i < tpc * E; i += kWarps * 32) {
            const int tl = i / E, e = i % E;
            float s = 0.f;
            for (int src = 0; src < kCS; ++src) s = __fadd_rn(s, sm.red[(size_t)(src * tpc + tl) * E + e]);
            sm.sc[tl * E + e] = (uint16_t)f32_to_bf16_bits(s);
        }
        __syncthreads();
        for (int tl = warp; tl < tpc; tl += kWarps) {
            const int t = t0 + rank * tpc + tl;
            if (t >= a.T) continue;
            const uint16_t* sr = sm.sc + tl * E;
            uint32_t cand[8];  // keys of this lane's experts e = lane + 32 i
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int e = lane + 32 * i;
                cand[i] = (e < E) ? ((order_key16(sr[e]) << 16) | (0xFFFFu - (uint32_t)e)) : 0u;
            }
            int my_idx = 0;
            float my_s = 0.f, top_s = 0.f;
            for (int j = 0; j < k; ++j) {
                uint32_t best = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) best = max(best, cand[i]);
                const uint32_t win = __reduce_max_sync(0xffffffffu, best);
                const int e = (int)(0xFFFFu - (win & 0xFFFFu));
                const float s = bf16_bits_to_f32(key16_to_bits(win >> 16));
                if (j == 0) top_s = s;
                if (lane == j) {
                    my_idx = e;
                    my_s = s;
                }
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (cand[i] == win) cand[i] = 0u;
            }
            const float ex = (lane < k) ? expf(__fsub_rn(my_s, top_s)) : 0.f;
            float sum = 0.f;
            for (int j = 0; j < k; ++j) sum = __fadd_rn(sum, __shfl_sync(0xffffffffu, ex, j));
            if (lane < k) {
                const float p = bf16_bits_to_f32(f32_to_bf16_bits(__fdiv_rn(ex, sum)));
                const float pes = bf16_bits_to_f32(pes_s[my_idx]);
                a.idx[(size_t)t * k + lane] = my_idx;
                a.w[(size_t)t * k + lane] = (uint16_t)f32_to_bf16_bits(__fmul_rn(p, pes));
            }
        }
        __syncwarp();
        __syncthreads();  // sc and red are read; the next tile may overwrite them
    }
    // The last tile's activation copies (if any were issued without a tile
    // to use them) cannot be pending: loads are issued only for tiles walked.
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------------
// Row router: the same computation as router_kernel, one CTA per 16 tokens
// over the whole hidden dimension, no cluster. The CTA keeps its 16 x rows
// in shared memory (H / 64 boxes of 16 rows x 128 B, the MMA's K-major
// layout) with the router_scale (and pre_w) row, sums each token's squares
// itself (warp w <-> token w: each lane takes every 32nd 16-byte chunk, four
// at a time into four two-float accumulators, merged by error-free
// two-sums, so the mean is the exactly rounded one as above), normalises in
// place with the same three bf16 roundings, and streams the router weight
// through a ring of stages of two 64-wide K blocks (128 experts x 128 B
// each, TMA) into one accumulator: D[e][t] in 16 TMEM columns. The scores leave
// TMEM by lane quarter, are rounded to bf16 and staged as [token][expert];
// warp w then takes token w's top k, softmax and per-expert scale as the
// cluster router does. No cross-CTA exchange or barrier: the tile's latency
// is its x copy, two passes over shared memory and the weight stream.
namespace {
constexpr int kRowTT = 16;                 // tokens a CTA (one warp each)
constexpr int kRowWarps = 16;
constexpr int kRowWStages = 4;             // most router-weight ring stages (two 64-wide K blocks each)
constexpr int kRowStageBytes = 2 * kWBlockBytes;
static_assert(kRowTT == kRowWarps, "warp w owns token w");
}  // namespace

// Router-weight ring stages that fit beside the x tile, the scores and the
// router_scale and pre_w rows (0 if fewer than 2).
__host__ __device__ inline int row_wstages(int H) {
    const long fixed = 1024 + (long)(H / 64) * kRowTT * 128 + (long)kRowTT * kChunkE * 2 + 4L * H;
    const long n = ((long)(232448 - 1024) - fixed) / kRowStageBytes;
    return n < 2 ? 0 : (n > kRowWStages ? kRowWStages : (int)n);
}

size_t router_rows_smem_bytes(int H) {
    const size_t nkb = (size_t)H / 64;
    return 1024 + nkb * kRowTT * 128 + (size_t)row_wstages(H) * kRowStageBytes + (size_t)kRowTT * kChunkE * 2 +
           4 * (size_t)H;
}

__global__ void __launch_bounds__(kRowWarps * 32, 1) router_rows_kernel(const __grid_constant__ CUtensorMap wmap,
                                                                        const __grid_constant__ CUtensorMap xmap,
                                                                        RouterArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ uint64_t xfull, mdone, wfull[kRowWStages], wempty[kRowWStages];
    __shared__ uint32_t tmem_base;
    __shared__ uint16_t pes_s[kChunkE];
    __shared__ float rs_s[kRowTT];
    __shared__ int abort_flag_s, have_s, got_s;
    pdl_trigger();
    pdl_wait();
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int H = a.H, E = a.E, k = a.k;
    const int nkb = H / 64;
    uint8_t* xt = base;                                             // nkb boxes of 16 rows x 128 B
    const int NW = row_wstages(H);                                  // weight ring stages
    const int nst = (nkb + 1) / 2;                                  // weight stages: K blocks 2s, 2s + 1
    uint8_t* wring = xt + (size_t)nkb * kRowTT * 128;               // NW stages of two 128-row x 128 B blocks
    uint16_t* sc = reinterpret_cast<uint16_t*>(wring + (size_t)NW * kRowStageBytes);  // [16][E]
    uint16_t* scl = sc + kRowTT * E;                                // router_scale [H]
    uint16_t* pwl = scl + H;                                        // pre_w [H] (expert input only)
    volatile int* abort_flag = &abort_flag_s;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = blockIdx.x * kRowTT;
    const uint32_t wbytes = (uint32_t)E * 128u;                     // one K block of the weight (E <= 128 rows)
    const int nw0 = nst < NW ? nst : NW;

    for (int e = threadIdx.x; e < E; e += blockDim.x) pes_s[e] = a.per_expert_scale[e];
    if (threadIdx.x == 0) {
        prefetch_tensormap(&xmap);
        prefetch_tensormap(&wmap);
        mbar_init(&xfull, 1);
        mbar_init(&mdone, 1);
        for (int s = 0; s < kRowWStages; ++s) {
            mbar_init(&wfull[s], 1);
            mbar_init(&wempty[s], 1);
        }
        abort_flag_s = 0;
        fence_barrier_init();
    }
    if (warp == 1) {  // scores accumulator: 128 lanes (experts) x 16 columns (tokens)
        tmem_alloc(&tmem_base, 32);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    if (threadIdx.x == 0) {
        // the tile's rows (rows past T read as zero), the router_scale (and
        // pre_w) row, and the first weight stages
        const uint32_t vbytes = (uint32_t)H * 2u;
        mbar_arrive_expect_tx(&xfull, (uint32_t)nkb * kRowTT * 128u + (a.xe ? 2u : 1u) * vbytes);
        for (int kb = 0; kb < nkb; ++kb) tma_load_2d(xt + (size_t)kb * kRowTT * 128, &xmap, &xfull, kb * 64, t0);
        bulk_load(scl, a.router_scale, vbytes, &xfull);
        if (a.xe) bulk_load(pwl, a.pre_w, vbytes, &xfull);
        for (int s = 0; s < nw0; ++s) {
            const int nb = min(2, nkb - 2 * s);
            mbar_arrive_expect_tx(&wfull[s], (uint32_t)nb * wbytes);
            for (int b = 0; b < nb; ++b)
                tma_load_2d(wring + (size_t)s * kRowStageBytes + (size_t)b * kWBlockBytes, &wmap, &wfull[s],
                            (2 * s + b) * 64, 0);
        }
    }
    if (warp == 0) {
        const bool h = mbar_wait(&xfull, 0, abort_flag);
        if (lane == 0) have_s = h;
    }
    __syncthreads();
    const bool have = have_s != 0;

    // ---- 1. sums of squares and 1/rms: warp w <-> token w ----
    {
        const int t = warp;
        const int nchunk = have ? nkb * 8 : 0;
        // four chunks a lane at a time into four two-float accumulators
        // (four independent chains), merged by two-sums at the end
        float hh[4] = {0.f, 0.f, 0.f, 0.f}, ll[4] = {0.f, 0.f, 0.f, 0.f};
        for (int i0 = lane; i0 < nchunk; i0 += 128) {
            uint32_t w[4][4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + 32 * u;
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (i < nchunk) v = *reinterpret_cast<const uint4*>(xt + (size_t)(i >> 3) * kRowTT * 128 + sw128(t, i & 7));
                w[u][0] = v.x;
                w[u][1] = v.y;
                w[u][2] = v.z;
                w[u][3] = v.w;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    // squares of bf16 values are exact in fp32 (zero chunks add nothing)
                    const float x0 = bf16_bits_to_f32(w[u][j] & 0xFFFFu), x1 = bf16_bits_to_f32(w[u][j] >> 16);
                    acc2(hh[u], ll[u], __fmul_rn(x0, x0));
                    acc2(hh[u], ll[u], __fmul_rn(x1, x1));
                }
            }
        }
        float hs, ls, se, ha, la, hb, lb;
        two_sum(hh[0], hh[1], ha, se);
        la = __fadd_rn(__fadd_rn(ll[0], ll[1]), se);
        two_sum(hh[2], hh[3], hb, se);
        lb = __fadd_rn(__fadd_rn(ll[2], ll[3]), se);
        two_sum(ha, hb, hs, se);
        ls = __fadd_rn(__fadd_rn(la, lb), se);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float h2 = __shfl_xor_sync(0xffffffffu, hs, o), l2 = __shfl_xor_sync(0xffffffffu, ls, o);
            float s2, e2;
            two_sum(hs, h2, s2, e2);
            hs = s2;
            ls = __fadd_rn(__fadd_rn(ls, l2), e2);
        }
        if (lane == 0) {
            // mean = (hs + ls) / H rounded once to fp32, as in router_kernel
            const float Hf = (float)H;
            const float q0 = __fdiv_rn(hs, Hf);
            const float rsd = __fadd_rn(__fmaf_rn(-q0, Hf, hs), ls);
            const float mean = __fadd_rn(q0, __fdiv_rn(rsd, Hf));
            rs_s[t] = __frsqrt_rn(__fadd_rn(mean, a.eps));
        }
    }
    __syncthreads();

    // ---- 2. normalise in place: element i is token i % 16, chunk i / 16 ----
    const uint32_t rootb = f32_to_bf16_bits(a.root), root2 = rootb | (rootb << 16);
    for (int i = threadIdx.x; have && i < kRowTT * nkb * 8; i += kRowWarps * 32) {
        const int t = i & (kRowTT - 1), c = i >> 4;
        const float rs = rs_s[t];
        uint4* p = reinterpret_cast<uint4*>(xt + (size_t)(c >> 3) * kRowTT * 128 + sw128(t, c & 7));
        const uint4 v = *p;
        const size_t h = (size_t)c * 8;  // first of the chunk's 8 hidden columns
        if (a.xe && t0 + t < a.T) {  // the expert input: bf16((x * rs) * pre_w), one rounding
            const uint4 pw = *reinterpret_cast<const uint4*>(pwl + h);
            const uint32_t xv[4] = {v.x, v.y, v.z, v.w}, wv[4] = {pw.x, pw.y, pw.z, pw.w};
            uint32_t e[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                e[j] = pack_bf16x2(
                    __fmul_rn(__fmul_rn(__uint_as_float(xv[j] << 16), rs), __uint_as_float(wv[j] << 16)),
                    __fmul_rn(__fmul_rn(__uint_as_float(xv[j] & 0xFFFF0000u), rs), __uint_as_float(wv[j] & 0xFFFF0000u)));
            *reinterpret_cast<uint4*>(a.xe + (size_t)(t0 + t) * H + h) = make_uint4(e[0], e[1], e[2], e[3]);
        }
        const uint4 sv = *reinterpret_cast<const uint4*>(scl + h);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w}, sw[4] = {sv.x, sv.y, sv.z, sv.w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t n = pack_bf16x2(__fmul_rn(__uint_as_float(w[j] << 16), rs),
                                           __fmul_rn(__uint_as_float(w[j] & 0xFFFF0000u), rs));
            o[j] = mul_bf16x2(mul_bf16x2(n, sw[j]), root2);
        }
        *p = make_uint4(o[0], o[1], o[2], o[3]);
    }
    // The normalised tile was written by ordinary stores; the tensor core
    // reads it through the async proxy.
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();

    // ---- 3. scores: D[e][t] += W[e][kb] . n[t][kb] over the K blocks ----
    // Warp 1's elected thread waits for each weight stage (two K blocks)
    // and issues its 8 MMAs in K order, whose commit frees the slot; warp 2
    // refills each freed slot with the stage NW further on, so NW - 1 or NW
    // stages stay in flight.
    if (warp == 1) {
        tc_fence_after();
        if (elect_one()) {
            const uint32_t idesc = idesc_bf16_m128((uint32_t)kRowTT);
            bool ok = have;
            for (int st = 0; ok && st < nst; ++st) {
                const int slot = st % NW;
                if (!(ok = mbar_wait(&wfull[slot], (uint32_t)(st / NW) & 1u, abort_flag))) break;
                tc_fence_after();
                for (int b = 0; b < 2 && 2 * st + b < nkb; ++b) {
                    const int kb = 2 * st + b;
                    const uint64_t ad = sw128_kmajor_desc(
                        smem_u32(wring + (size_t)slot * kRowStageBytes + (size_t)b * kWBlockBytes));
                    const uint64_t bd = sw128_kmajor_desc(smem_u32(xt + (size_t)kb * kRowTT * 128));
#pragma unroll
                    for (int k16 = 0; k16 < 4; ++k16)
                        umma_ss(tmem, ad + (uint64_t)(k16 * 2), bd + (uint64_t)(k16 * 2), idesc,
                                (kb > 0 || k16 > 0) ? 1u : 0u);
                }
                umma_commit(&wempty[slot]);
            }
            umma_commit(&mdone);  // every MMA above (none if the tile was not loaded)
        }
        __syncwarp();
    } else if (warp == 2) {
        if (elect_one()) {
            int issued = nw0;  // weight stages whose copies have been issued
            for (int st = nw0; have && st < nst; ++st) {
                const int slot = st % NW;
                if (!mbar_wait(&wempty[slot], (uint32_t)((st - NW) / NW) & 1u, abort_flag)) break;
                const int nb = min(2, nkb - 2 * st);
                mbar_arrive_expect_tx(&wfull[slot], (uint32_t)nb * wbytes);
                for (int b = 0; b < nb; ++b)
                    tma_load_2d(wring + (size_t)slot * kRowStageBytes + (size_t)b * kWBlockBytes, &wmap, &wfull[slot],
                                (2 * st + b) * 64, 0);
                issued = st + 1;
            }
            // The last copies issued into each slot land before the CTA
            // exits (earlier ones were consumed by the MMAs before the slot
            // was refilled).
            for (int st = issued - 1; st >= 0 && st >= issued - NW; --st)
                mbar_drain(&wfull[st % NW], (uint32_t)(st / NW) & 1u);
        }
        __syncwarp();
    }
    if (warp == 0) {
        const bool g = mbar_wait(&mdone, 0, abort_flag);
        if (lane == 0) got_s = g && have;
    }
    __syncthreads();
    tc_fence_after();
    const bool got = got_s != 0;

    // ---- 4. scores to shared memory as [token][expert] bf16 ----
    if (warp < 4) {
        uint32_t v[16];
        if (got) {
            tmem_ld16(tmem + ((uint32_t)(32 * warp) << 16), v);
            tmem_wait_ld();
        } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = 0u;
        }
        const int e = 32 * warp + lane;
        if (e < E) {
#pragma unroll
            for (int j = 0; j < kRowTT; ++j) sc[j * E + e] = (uint16_t)f32_to_bf16_bits(__uint_as_float(v[j]));
        }
    }
    tc_fence_before();
    __syncthreads();

    // ---- 5. token warp: top k, precise softmax, per-expert scale ----
    const int t = t0 + warp;
    if (got && t < a.T) {
        const uint16_t* sr = sc + warp * E;
        uint32_t cand[4];  // keys of this lane's experts e = lane + 32 i (E <= 128)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int e = lane + 32 * i;
            cand[i] = (e < E) ? ((order_key16(sr[e]) << 16) | (0xFFFFu - (uint32_t)e)) : 0u;
        }
        int my_idx = 0;
        float my_s = 0.f, top_s = 0.f;
        for (int j = 0; j < k; ++j) {
            uint32_t best = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) best = max(best, cand[i]);
            const uint32_t win = __reduce_max_sync(0xffffffffu, best);
            const int e = (int)(0xFFFFu - (win & 0xFFFFu));
            const float sv = bf16_bits_to_f32(key16_to_bits(win >> 16));
            if (j == 0) top_s = sv;
            if (lane == j) {
                my_idx = e;
                my_s = sv;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (cand[i] == win) cand[i] = 0u;
        }
        const float ex = (lane < k) ? expf(__fsub_rn(my_s, top_s)) : 0.f;
        float sum = 0.f;
        for (int j = 0; j < k; ++j) sum = __fadd_rn(sum, __shfl_sync(0xffffffffu, ex, j));
        if (lane < k) {
            const float pr = bf16_bits_to_f32(f32_to_bf16_bits(__fdiv_rn(ex, sum)));
            const float pes = bf16_bits_to_f32(pes_s[my_idx]);
            a.idx[(size_t)t * k + lane] = my_idx;
            a.w[(size_t)t * k + lane] = (uint16_t)f32_to_bf16_bits(__fmul_rn(pr, pes));
        }
    }
    if (!have && threadIdx.x == 0) mbar_drain(&xfull, 0);  // the tile's copies land before exit
    __syncwarp();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 32);
    }
}

int router_error_word() {
    int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_error_word, sizeof(int)) != cudaSuccess) return 0;
    cudaMemcpyToSymbol(g_error_word, &z, sizeof(int));
    return v;
}

namespace {
constexpr size_t kRouterSmemLimit = 232448 - 1024;  // 227 KB per CTA minus the static part
}

size_t router_smem_bytes(int H, int E, int tt) { return 1024 + router_layout(H, E, tt, nullptr, nullptr); }

namespace {
cudaError_t ensure_router_attr() {
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        cudaError_t err = cudaFuncSetAttribute(router_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)kRouterSmemLimit);
        if (err != cudaSuccess) return err;
        attr_set[dev] = true;
    }
    return cudaSuccess;
}

cudaLaunchConfig_t router_config(int clusters, size_t smem, cudaStream_t stream, cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(clusters * kCS), 1, 1);
    cfg.blockDim = dim3(kWarps * 32, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kCS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cfg;
}

// Clusters of this kernel the device holds at once with `smem` bytes per CTA
// (cached per device and size).
int router_resident_clusters(size_t smem) {
    static std::mutex mu;
    static std::map<std::pair<int, size_t>, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || ensure_router_attr() != cudaSuccess) return 1;
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find({dev, smem});
    if (it != cache.end()) return it->second;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = router_config(1, smem, nullptr, attr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, router_kernel, &cfg) != cudaSuccess || n < 1) n = 1;
    cache[{dev, smem}] = n;
    return n;
}
}  // namespace

// Tokens per cluster: the smallest of 16, 32, 64 whose clusters all fit on
// the device at once (one wave); the largest that fits in shared memory when
// none does.
int router_tokens_per_cluster(int T, int H, int E) {
    int best = 16;
    for (int tt = 16; tt <= 64; tt <<= 1) {
        const size_t smem = router_smem_bytes(H, E, tt);
        if (smem > kRouterSmemLimit) break;
        best = tt;
        if ((T + tt - 1) / tt <= router_resident_clusters(smem)) return tt;
    }
    return best;
}

cudaError_t launch_router(const CUtensorMap& wmap, const CUtensorMap& xmap, const RouterArgs& a,
                          cudaStream_t stream) {
    if (a.T == 0) return cudaSuccess;
    const size_t smem = router_smem_bytes(a.H, a.E, a.tt);
    if (smem > kRouterSmemLimit || a.tt % 16 != 0 || a.tt > 64) return cudaErrorInvalidValue;
    cudaError_t err = ensure_router_attr();
    if (err != cudaSuccess) return err;
    // Persistent clusters: as many as the device holds at once, at most one
    // per token tile; each walks its share of the tiles.
    const int ntiles = (a.T + a.tt - 1) / a.tt;
    const int clusters = std::min(ntiles, router_resident_clusters(smem));
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = router_config(clusters, smem, stream, attr);
    return cudaLaunchKernelEx(&cfg, router_kernel, wmap, xmap, a);
}

namespace {
cudaError_t ensure_router_rows_attr() {
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        cudaError_t err = cudaFuncSetAttribute(router_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)kRouterSmemLimit);
        if (err != cudaSuccess) return err;
        attr_set[dev] = true;
    }
    return cudaSuccess;
}
}  // namespace

bool router_rows_fits(int H, int E, bool q4) {
    return !q4 && E >= 1 && E <= kChunkE && H % 64 == 0 && H >= 64 && row_wstages(H) >= 2 &&
           router_rows_smem_bytes(H) <= kRouterSmemLimit;
}

// The row router where it fits and the cluster router would walk two or
// more waves of tiles. Measured at H = 2816, E = 128 (us, launch included,
// L2 flushed): one wave of row-router CTAs takes ~23 us whatever T, while a
// cluster takes ~6 us a tile after ~3 us of setup: T = 256: cluster 15.0,
// row 23.1; T = 512 and 768 (one wave): 17.0 / 23.2; T = 1024 and 1536 (two
// waves): 25.2 / 23.2; T = 2048 (three): 33.4 / 23.7; T = 4096 (five):
// 47.7 / 41.6.
bool router_prefer_rows(int T, int H, int E) {
    if (!router_rows_fits(H, E, false)) return false;
    const int tt = router_tokens_per_cluster(T, H, E);
    const size_t smem = router_smem_bytes(H, E, tt);
    if (smem > kRouterSmemLimit) return true;
    const int waves = ((T + tt - 1) / tt + router_resident_clusters(smem) - 1) / router_resident_clusters(smem);
    return waves >= 2;
}

cudaError_t launch_router_rows(const CUtensorMap& wmap, const CUtensorMap& xmap, const RouterArgs& a,
                               cudaStream_t stream) {
    if (a.T == 0) return cudaSuccess;
    if (!router_rows_fits(a.H, a.E, a.rq_w != nullptr) || a.k < 1 || a.k > 32 || a.k > a.E) return cudaErrorInvalidValue;
    cudaError_t err = ensure_router_rows_attr();
    if (err != cudaSuccess) return err;
    const int ctas = (a.T + kRowTT - 1) / kRowTT;
    return launch_pdl(router_rows_kernel, dim3((unsigned)ctas), dim3(kRowWarps * 32), router_rows_smem_bytes(a.H),
                      stream, wmap, xmap, a);
}

}  // namespace moe
