// Router kernel: DiffRouter.forward of the DiffusionGemma language model
// ("diffusion-gemma/model.ts"), fused into one launch.
//
// One thread-block cluster handles 16 tokens; its CS = ceil(E/32) CTAs each
// own 32 experts. In every CTA a producer warp brings, by TMA with the
// 128-byte swizzle, the 16 x H activation tile (16-row x 64-column boxes)
// and, through an 8-deep ring, 64-wide K blocks of its 32 router-weight rows.
// Four compute warps
//   1. apply the no-scale RMS norm in fp32 to the tile in shared memory, in
//      place (the fp32 semantics are the ones "diffusion-gemma/vision.ts"
//      spells out in manualRms), followed by the two bf16 multiplies (router
//      scale, H^-0.5);
//   2. compute 16 tokens x 32 experts of scores with mma.sync m16n8k16 (fp32
//      accumulate), round them to bf16 and write them into the leader CTA's
//      shared memory (distributed shared memory);
// then the leader CTA picks the top k per token (value descending, ties to
// the lower expert id), takes the fp32 softmax over the k picked scores and
// multiplies by per_expert_scale[idx].
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"

namespace cg = cooperative_groups;

namespace moe {

namespace {

constexpr int kTT = 16;        // tokens per cluster
constexpr int kWarps = 4;      // compute warps per CTA (+1 producer warp)
constexpr int kExpPerCta = 32; // experts per CTA (8 per warp)
constexpr int kRing = 8;       // K blocks of router weight in flight
constexpr int kBlockBytes = kExpPerCta * 128;  // 32 rows x 64 bf16
constexpr int kXBoxBytes = kTT * 128;          // 16 rows x 64 bf16

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// bf16 bits -> key that orders like the value (for finite values).
__device__ __forceinline__ uint32_t order_key16(uint32_t b) { return (b & 0x8000u) ? (~b & 0xFFFFu) : (b | 0x8000u); }
__device__ __forceinline__ uint32_t key16_to_bits(uint32_t k) { return (k & 0x8000u) ? (k & 0x7FFFu) : (~k & 0xFFFFu); }

// Byte offset of 16-byte chunk c (0..7) of row r inside a 128-byte-swizzled
// box of 128-byte rows.
__device__ __forceinline__ int sw128(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

}  // namespace

__global__ void __launch_bounds__((kWarps + 1) * 32) router_kernel(const __grid_constant__ CUtensorMap wmap,
                                                                    const __grid_constant__ CUtensorMap xmap,
                                                                    RouterArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ uint64_t full[kRing], empty[kRing], xfull;
    __shared__ int abort_flag_s;
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int H = a.H, E = a.E, k = a.k;
    const int nkb = H / 64;
    uint8_t* ring = smem;                      // kRing x 4 KB
    uint8_t* xt = smem + kRing * kBlockBytes;  // nkb boxes of 16 rows x 128 B (swizzled)
    uint16_t* rscale = reinterpret_cast<uint16_t*>(xt + nkb * kXBoxBytes);  // router_scale [H]
    uint16_t* scores = rscale + H;                                             // [kTT][E], leader CTA
    volatile int* abort_flag = &abort_flag_s;

    cg::cluster_group cluster = cg::this_cluster();
    const int cs = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();
    const int t0 = (blockIdx.x / cs) * kTT;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kRing; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kWarps);
        }
        mbar_init(&xfull, 1);
        abort_flag_s = 0;
        fence_barrier_init();
    }
    // All CTAs of the cluster have started (and initialised their barriers)
    // before any of them writes into the leader's shared memory.
    cluster_barrier();

    if (warp == kWarps) {
        // ---- producer ----
        if (lane == 0) {
            prefetch_tensormap(&xmap);
            prefetch_tensormap(&wmap);
            mbar_arrive_expect_tx(&xfull, nkb * kXBoxBytes + H * 2);
            bulk_load(rscale, a.router_scale, H * 2, &xfull);
            for (int kb = 0; kb < nkb; ++kb) tma_load_2d(xt + kb * kXBoxBytes, &xmap, &xfull, kb * 64, t0);
            int kb = 0;
            for (; kb < nkb; ++kb) {
                const int slot = kb % kRing;
                if (!mbar_wait(&empty[slot], ((kb / kRing) & 1) ^ 1, abort_flag)) break;
                mbar_arrive_expect_tx(&full[slot], kBlockBytes);
                tma_load_2d(ring + slot * kBlockBytes, &wmap, &full[slot], kb * 64, rank * kExpPerCta);
            }
            // no copies in flight at exit
            mbar_wait(&xfull, 0, abort_flag);
            for (int b = (kb > kRing ? kb - kRing : 0); b < kb; ++b) mbar_wait(&full[b % kRing], (b / kRing) & 1, abort_flag);
        }
        __syncwarp();
        cluster_barrier();
        return;
    }

    // ---- 1. no-scale RMS norm, x scale, x H^-0.5 (bf16 after each op), in place ----
    const bool have_x = mbar_wait(&xfull, 0, abort_flag);
    const int nchunks = nkb * 8;  // 16-byte chunks per row
    for (int r = warp; r < kTT && have_x; r += kWarps) {
        float ss = 0.f;
#pragma unroll 4
        for (int i = lane; i < nchunks; i += 32) {
            const uint4 v = *reinterpret_cast<const uint4*>(xt + (i >> 3) * kXBoxBytes + sw128(r, i & 7));
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float lo = bf16_bits_to_f32(w[j] & 0xFFFFu), hi = bf16_bits_to_f32(w[j] >> 16);
                ss = __fadd_rn(ss, __fmul_rn(lo, lo));
                ss = __fadd_rn(ss, __fmul_rn(hi, hi));
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
        const float rs = __frsqrt_rn(__fadd_rn(__fdiv_rn(ss, (float)H), a.eps));
#pragma unroll 4
        for (int i = lane; i < nchunks; i += 32) {
            uint4* p = reinterpret_cast<uint4*>(xt + (i >> 3) * kXBoxBytes + sw128(r, i & 7));
            const uint4 v = *p;
            const uint4 s = reinterpret_cast<const uint4*>(rscale)[i];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w}, sc[4] = {s.x, s.y, s.z, s.w};
            uint32_t o[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float n_lo = bf16_bits_to_f32(f32_to_bf16_bits(__fmul_rn(bf16_bits_to_f32(w[j] & 0xFFFFu), rs)));
                float n_hi = bf16_bits_to_f32(f32_to_bf16_bits(__fmul_rn(bf16_bits_to_f32(w[j] >> 16), rs)));
                n_lo = bf16_bits_to_f32(f32_to_bf16_bits(__fmul_rn(n_lo, bf16_bits_to_f32(sc[j] & 0xFFFFu))));
                n_hi = bf16_bits_to_f32(f32_to_bf16_bits(__fmul_rn(n_hi, bf16_bits_to_f32(sc[j] >> 16))));
                o[j] = pack_bf16x2(__fmul_rn(n_lo, a.root), __fmul_rn(n_hi, a.root));
            }
            *p = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
    // The compute warps only (the producer warp never comes here): named
    // barrier 1 over kWarps * 32 threads.
    asm volatile("bar.sync 1, %0;" ::"n"(kWarps * 32) : "memory");

    // ---- 2. scores for experts [e0, e0+8) of this warp: 16 tokens x 8 experts ----
    // Inside each 64-wide K block, thread (g, q) owns K [16q, 16q+16) of its
    // rows (chunks 2q and 2q+1); mma step s takes K 16q+4s+{0,1} as fragment
    // k {2q, 2q+1} and 16q+4s+{2,3} as k {2q+8, 2q+9}, identically for both
    // operands, so the four steps sum the block's 64 products exactly once.
    const int e0 = rank * kExpPerCta + warp * 8;
    const int g = lane >> 2, q = lane & 3;
    const int brow = warp * 8 + g;  // row of this lane's expert in a ring block
    float c[4] = {0.f, 0.f, 0.f, 0.f};
    for (int kb = 0; kb < nkb && have_x; ++kb) {
        const int slot = kb % kRing;
        if (!mbar_wait(&full[slot], (kb / kRing) & 1, abort_flag)) break;
        const uint8_t* blk = ring + slot * kBlockBytes;
        const uint4 b0 = *reinterpret_cast<const uint4*>(blk + sw128(brow, 2 * q));
        const uint4 b1 = *reinterpret_cast<const uint4*>(blk + sw128(brow, 2 * q + 1));
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
        const uint8_t* xb = xt + kb * kXBoxBytes;
        const uint4 x0 = *reinterpret_cast<const uint4*>(xb + sw128(g, 2 * q));
        const uint4 x1 = *reinterpret_cast<const uint4*>(xb + sw128(g, 2 * q + 1));
        const uint4 y0 = *reinterpret_cast<const uint4*>(xb + sw128(g + 8, 2 * q));
        const uint4 y1 = *reinterpret_cast<const uint4*>(xb + sw128(g + 8, 2 * q + 1));
        const uint32_t ar0[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        const uint32_t ar1[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
        const uint32_t br[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
        for (int s = 0; s < 4; ++s)
            mma_bf16_16816(c, ar0[2 * s], ar1[2 * s], ar0[2 * s + 1], ar1[2 * s + 1], br[2 * s], br[2 * s + 1]);
    }
    // c0,c1: token g, experts e0+2q, e0+2q+1; c2,c3: token g+8.
    uint16_t* lead = cluster.map_shared_rank(scores, 0);
    {
        const int ea = e0 + 2 * q;
        if (ea < E) {
            lead[g * E + ea] = (uint16_t)f32_to_bf16_bits(c[0]);
            lead[(g + 8) * E + ea] = (uint16_t)f32_to_bf16_bits(c[2]);
        }
        if (ea + 1 < E) {
            lead[g * E + ea + 1] = (uint16_t)f32_to_bf16_bits(c[1]);
            lead[(g + 8) * E + ea + 1] = (uint16_t)f32_to_bf16_bits(c[3]);
        }
    }
    __syncwarp();
    cluster_barrier();
    if (rank != 0) return;

    // ---- 3. top-k + precise softmax + per-expert scale (leader CTA) ----
    for (int tl = warp; tl < kTT; tl += kWarps) {
        const int t = t0 + tl;
        if (t >= a.T) continue;
        const uint16_t* sr = scores + tl * E;
        uint32_t cand[8];  // keys of this lane's experts e = lane + 32 i
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = lane + 32 * i;
            cand[i] = (e < E) ? ((order_key16(sr[e]) << 16) | (0xFFFFu - (uint32_t)e)) : 0u;
        }
        int my_idx = 0;
        float my_s = 0.f;
        float top_s = 0.f;
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
            const float pes = bf16_bits_to_f32(a.per_expert_scale[my_idx]);
            a.idx[(size_t)t * k + lane] = my_idx;
            a.w[(size_t)t * k + lane] = (uint16_t)f32_to_bf16_bits(__fmul_rn(p, pes));
        }
    }
}

int router_error_word() {
    int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_error_word, sizeof(int)) != cudaSuccess) return 0;
    cudaMemcpyToSymbol(g_error_word, &z, sizeof(int));
    return v;
}

size_t router_smem_bytes(int H, int E) {
    return 1024 + (size_t)kRing * kBlockBytes + (size_t)(H / 64) * kXBoxBytes + (size_t)H * 2 + (size_t)kTT * E * 2;
}

cudaError_t launch_router(const CUtensorMap& wmap, const CUtensorMap& xmap, const RouterArgs& a,
                          cudaStream_t stream) {
    if (a.T == 0) return cudaSuccess;
    const int cs = (a.E + kExpPerCta - 1) / kExpPerCta;
    const int tiles = (a.T + kTT - 1) / kTT;
    const size_t smem = router_smem_bytes(a.H, a.E);
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        cudaError_t err = cudaFuncSetAttribute(router_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448 - 1024);
        if (err != cudaSuccess) return err;
        attr_set[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(tiles * cs, 1, 1);
    cfg.blockDim = dim3((kWarps + 1) * 32, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, router_kernel, wmap, xmap, a);
}

}  // namespace moe
