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
    for (int e = tid; e < E; e += kDispatchThreads) {
        int run = 0;
        for (int w = 0; w < kW; ++w) {
            const int v = wh[w][e];
            wh[w][e] = run;
            run += v;
        }
        cnt[e] = run;
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
        if (tid == 0 && a.num_tiles) {
            int mx = 0;
            for (int e = 0; e < E; ++e) mx = max(mx, min(cnt[e], a.nmax));
            a.num_tiles[0] = tbase[E];
            a.num_tiles[1] = mx;  // rows of the largest token tile
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
    dispatch_kernel<<<1, kDispatchThreads, 0, stream>>>(a);
    return cudaGetLastError();
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

__global__ void gather_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ perm,
                              const int32_t* __restrict__ offsets, uint16_t* __restrict__ xs, int S, int k,
                              int H, int E) {
    const int chunks = H / 8;
    const int valid = offsets[E];
    const long total = (long)S * chunks;
    for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total; i += (long)gridDim.x * blockDim.x) {
        const int p = (int)(i / chunks), c = (int)(i % chunks);
        if (p >= valid) continue;
        const int t = perm[p] / k;
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + (size_t)t * H) + c);
        reinterpret_cast<uint4*>(xs + (size_t)p * H)[c] = interleave8(v);
    }
}

cudaError_t launch_gather(const uint16_t* x, const int32_t* perm, const int32_t* offsets, uint16_t* xs,
                          int S, int k, int H, int E, cudaStream_t stream) {
    if (S == 0) return cudaSuccess;
    const long total = (long)S * (H / 8);
    const int threads = 256;
    long blocks = (total + threads - 1) / threads;
    if (blocks > 152 * 16) blocks = 152 * 16;
    gather_kernel<<<(int)blocks, threads, 0, stream>>>(x, perm, offsets, xs, S, k, H, E);
    return cudaGetLastError();
}

__global__ void combine_kernel(const uint16_t* __restrict__ y, const uint16_t* __restrict__ w,
                               uint16_t* __restrict__ out, int T, int k, int H) {
    const int chunks = H / 8;
    const long total = (long)T * chunks;
    for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total; i += (long)gridDim.x * blockDim.x) {
        const int t = (int)(i / chunks), c = (int)(i % chunks);
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int j = 0; j < k; ++j) {
            const size_t f = (size_t)t * k + j;
            const float wj = bf16_bits_to_f32(w[f]);
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(y + f * H) + c);
            const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float lo = bf16_bits_to_f32(f32_to_bf16_bits(__fmul_rn(bf16_bits_to_f32(u[q] & 0xFFFFu), wj)));
                const float hi = bf16_bits_to_f32(f32_to_bf16_bits(__fmul_rn(bf16_bits_to_f32(u[q] >> 16), wj)));
                acc[2 * q] = __fadd_rn(acc[2 * q], lo);
                acc[2 * q + 1] = __fadd_rn(acc[2 * q + 1], hi);
            }
        }
        uint4 o;
        o.x = pack_bf16x2(acc[0], acc[1]);
        o.y = pack_bf16x2(acc[2], acc[3]);
        o.z = pack_bf16x2(acc[4], acc[5]);
        o.w = pack_bf16x2(acc[6], acc[7]);
        reinterpret_cast<uint4*>(out + (size_t)t * H)[c] = o;
    }
}

cudaError_t launch_combine(const uint16_t* y, const uint16_t* w, uint16_t* out, int T, int k, int H,
                           cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const long total = (long)T * (H / 8);
    const int threads = 256;
    long blocks = (total + threads - 1) / threads;
    if (blocks > 152 * 16) blocks = 152 * 16;
    combine_kernel<<<(int)blocks, threads, 0, stream>>>(y, w, out, T, k, H);
    return cudaGetLastError();
}

int dispatch_error_word() {
    int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_error_word, sizeof(int)) != cudaSuccess) return 0;
    cudaMemcpyToSymbol(g_error_word, &z, sizeof(int));
    return v;
}

}  // namespace moe
