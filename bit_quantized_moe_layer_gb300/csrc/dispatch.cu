// Dispatch, gather and combine kernels of DiffExperts.forward
// ("diffusion-gemma/model.ts"):
//  - dispatch: the sorted path's argsort of the flat indices, its inverse and
//    rows = order // k, as a stable counting sort by expert id, plus the list
//    of per-expert token tiles the grouped GEMMs walk;
//  - gather: the sorted path's take of x rows (rowIdx), stored in the K order
//    the grouped GEMM's dequantised weights use;
//  - combine: the un-sort, (y * weights[..., None]).sum(-2), per token.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {
constexpr int kDispatchThreads = 1024;
constexpr int kMaxE = 256;
}  // namespace

// One CTA of 32 warps; warp w owns the contiguous slot range
// [w*per, (w+1)*per). Pass 1: per-warp histograms (warp match-any, one add
// per group of equal ids). Then per expert an exclusive scan over warps, a
// scan over experts (offsets and token-tile bases) and the tile list. Pass 2:
// each warp walks its range again in slot order and places each slot at its
// warp's running base for that expert plus its rank among equal ids in the
// 32-slot group. Warps cover the slots in order, so the sort is stable and
// the result unique.
__global__ void __launch_bounds__(kDispatchThreads) dispatch_kernel(DispatchArgs a) {
    constexpr int kW = kDispatchThreads / 32;
    __shared__ int wh[kW][kMaxE + 1];
    __shared__ int cnt[kMaxE], off[kMaxE + 1], tbase[kMaxE + 1];
    pdl_trigger();
    pdl_wait();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = a.S, E = a.E;
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int i = tid; i < kW * (kMaxE + 1); i += kDispatchThreads) (&wh[0][0])[i] = 0;
    __syncthreads();
    const int per = (S + kW - 1) / kW;
    const int c0 = min(S, warp * per), c1 = min(S, c0 + per);
    for (int b = c0; b < c1; b += 32) {
        const int f = b + lane;
        int e = (f < c1) ? a.idx[f] : -1;
        if (f < c1 && (e < 0 || e >= E)) {
            atomicOr(&g_error_word, kErrBadExpert);
            e = -1;
        }
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && (peers & lt_mask) == 0) wh[warp][e] += __popc(peers);
    }
    __syncthreads();
    // Per expert, exclusive scan over the 32 warps' counts: warp ww scans the
    // columns of experts ww, ww + 32, ..., lane = source warp.
    for (int e = warp; e < E; e += kW) {
        const int v = wh[lane][e];
        int inc = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += u;
        }
        wh[lane][e] = inc - v;
        if (lane == 31) cnt[e] = inc;
    }
    __syncthreads();
    if (warp == 0) {  // scan over experts: lane owns experts [8 lane, 8 lane + 8)
        int lc[8], lt[8], sc = 0, st = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int e = lane * 8 + j;
            lc[j] = (e < E) ? cnt[e] : 0;
            lt[j] = (lc[j] + a.nmax - 1) / a.nmax;
            sc += lc[j];
            st += lt[j];
        }
        int ic = sc, it = st;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int vc = __shfl_up_sync(0xffffffffu, ic, o), vt = __shfl_up_sync(0xffffffffu, it, o);
            if (lane >= o) {
                ic += vc;
                it += vt;
            }
        }
        int rc = ic - sc, rt = it - st;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int e = lane * 8 + j;
            if (e < E) {
                off[e] = rc;
                tbase[e] = rt;
            }
            rc += lc[j];
            rt += lt[j];
        }
        if (lane == 31) {
            off[E] = ic;
            tbase[E] = it;
        }
    }
    __syncthreads();
    for (int e = tid; e <= E; e += kDispatchThreads) a.offsets[e] = off[e];
    if (a.tiles) {
        for (int e = tid; e < E; e += kDispatchThreads) {
            for (int i = 0; tbase[e] + i < tbase[e + 1]; ++i) {
                Tile t;
                t.e = e;
                t.p0 = off[e] + i * a.nmax;
                t.rows = min(a.nmax, cnt[e] - i * a.nmax);
                t.pad = 0;
                a.tiles[tbase[e] + i] = t;
            }
        }
        if (warp == 0 && a.num_tiles) {
            int mx = 0;
            for (int e = lane; e < E; e += 32) mx = max(mx, min(cnt[e], a.nmax));
            mx = __reduce_max_sync(0xffffffffu, mx);
            if (lane == 0) {
                a.num_tiles[0] = tbase[E];
                a.num_tiles[1] = mx;  // rows of the largest token tile
            }
        }
    }
    for (int i = tid; i < kW * E; i += kDispatchThreads) wh[i / E][i % E] += off[i % E];
    __syncthreads();
    for (int b = c0; b < c1; b += 32) {
        const int f = b + lane;
        int e = (f < c1) ? a.idx[f] : -1;
        if (e >= E) e = -1;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(peers & lt_mask);
        if (e >= 0) {
            const int p = wh[warp][e] + rank;
            a.perm[p] = f;
            a.inv[f] = p;
        }
        __syncwarp();
        if (e >= 0 && rank == 0) wh[warp][e] += __popc(peers);
        __syncwarp();
    }
}

cudaError_t launch_dispatch(const DispatchArgs& a, cudaStream_t stream) {
    return launch_pdl(dispatch_kernel, dim3(1), dim3(kDispatchThreads), 0, stream, a);
}

// 8 bf16 (one 16-byte chunk) -> positions holding elements (0,4,1,5,2,6,3,7).
__device__ __forceinline__ uint4 interleave8(uint4 v) {
    uint4 o;
    o.x = __byte_perm(v.x, v.z, 0x5410);
    o.y = __byte_perm(v.x, v.z, 0x7632);
    o.z = __byte_perm(v.y, v.w, 0x5410);
    o.w = __byte_perm(v.y, v.w, 0x7632);
    return o;
}

// One warp per sorted row p: t = perm[p] / k, then the warp's lanes copy the
// row's 16-byte chunks (8 bf16 each), interleaved, lane-strided.
constexpr int kRowWarps = 8;  // rows (gather) or tokens (combine) per 256-thread block

__global__ void __launch_bounds__(kRowWarps * 32) gather_kernel(const uint16_t* __restrict__ x,
                                                                const int32_t* __restrict__ perm,
                                                                const int32_t* __restrict__ offsets,
                                                                uint16_t* __restrict__ xs, int S, int k, int H,
                                                                int E) {
    pdl_trigger();
    pdl_wait();
    const int p = blockIdx.x * kRowWarps + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (p >= S || p >= offsets[E]) return;
    const int t = perm[p] / k;
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H);
    uint4* dst = reinterpret_cast<uint4*>(xs + (size_t)p * H);
    const int chunks = H / 8;
#pragma unroll 4
    for (int c = lane; c < chunks; c += 32) dst[c] = interleave8(__ldg(src + c));
}

cudaError_t launch_gather(const uint16_t* x, const int32_t* perm, const int32_t* offsets, uint16_t* xs,
                          int S, int k, int H, int E, cudaStream_t stream) {
    if (S == 0) return cudaSuccess;
    return launch_pdl(gather_kernel, dim3((S + kRowWarps - 1) / kRowWarps), dim3(kRowWarps * 32), 0, stream, x, perm,
                      offsets, xs, S, k, H, E);
}

// One thread per (token t = blockIdx.x, 16-byte chunk c of H):
// out[t] = bf16(sum_j bf16(y[t k + j] * w[t k + j])), the products rounded to
// bf16 (the product of two bf16 arrays is a bf16 array) and summed in fp32
// in j order.
__global__ void __launch_bounds__(128) combine_kernel(const uint16_t* __restrict__ y,
                                                      const uint16_t* __restrict__ w,
                                                      uint16_t* __restrict__ out, int k, int H) {
    pdl_trigger();
    pdl_wait();
    const int chunks = H / 8;
    const int t = blockIdx.x, c = blockIdx.y * 128 + threadIdx.x;
    if (c >= chunks) return;
    const uint4* yt = reinterpret_cast<const uint4*>(y + (size_t)t * k * H) + c;
    const uint16_t* wt = w + (size_t)t * k;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (int j = 0; j < k; ++j) {
        const float wj = bf16_bits_to_f32(__ldg(wt + j));
        const uint4 v = __ldg(yt + (size_t)j * chunks);
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float lo = bf16_bits_to_f32(f32_to_bf16_bits(__fmul_rn(bf16_bits_to_f32(u[q] & 0xFFFFu), wj)));
            const float hi = bf16_bits_to_f32(f32_to_bf16_bits(__fmul_rn(bf16_bits_to_f32(u[q] >> 16), wj)));
            acc[2 * q] = __fadd_rn(acc[2 * q], lo);
            acc[2 * q + 1] = __fadd_rn(acc[2 * q + 1], hi);
        }
    }
    reinterpret_cast<uint4*>(out + (size_t)t * H)[c] =
        make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                   pack_bf16x2(acc[6], acc[7]));
}

cudaError_t launch_combine(const uint16_t* y, const uint16_t* w, uint16_t* out, int T, int k, int H,
                           cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const dim3 grid((unsigned)T, (unsigned)((H / 8 + 127) / 128));
    return launch_pdl(combine_kernel, grid, dim3(128), 0, stream, y, w, out, k, H);
}

int dispatch_error_word() {
    int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_error_word, sizeof(int)) != cudaSuccess) return 0;
    cudaMemcpyToSymbol(g_error_word, &z, sizeof(int));
    return v;
}

}  // namespace moe
