// Dispatch, gather and combine kernels of DiffExperts.forward
// ("diffusion-gemma/model.ts"):
//  - dispatch: the sorted path's argsort of the flat indices, its inverse and
//    rows = order // k, as a stable counting sort by expert id, plus the list
//    of per-expert token tiles the grouped GEMMs walk;
//  - gather: the sorted path's take of x rows (rowIdx), stored in the K order
//    the grouped GEMM's dequantised weights use;
//  - combine: the un-sort, (y * weights[..., None]).sum(-2), per token.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {
constexpr int kDispatchThreads = 1024;
constexpr int kW = kDispatchThreads / 32;
constexpr int kMaxE = 256;
constexpr int kFusedMaxRows = 64;  // sorted rows a CTA of the fused dispatch + gather writes

struct DispatchSmem {
    int wh[kW][kMaxE + 1];  // per-warp counts, then per-warp bases
    int cnt[kMaxE], off[kMaxE + 1], tbase[kMaxE + 1];
};

// The lanes of the warp whose expert id equals this lane's (e < 0 for a
// dropped or absent slot, which all match one another): the mask
// __match_any_sync would give, built from one ballot per bit of e + 1
// (bits = the bits of E), far cheaper than the match instruction here.
__device__ __forceinline__ unsigned same_expert_lanes(int e, int bits) {
    const unsigned v = (unsigned)(e + 1);
    unsigned peers = 0xffffffffu;
    for (int b = 0; b < bits; ++b) {
        const unsigned bit = (v >> b) & 1u;
        const unsigned m = __ballot_sync(0xffffffffu, bit != 0u);
        peers &= bit ? m : ~m;
    }
    return peers;
}

// Counts of the slots [c0, c1) by expert into wh_row (lanes of equal id: one add
// per group of equal ids). Out-of-range ids are dropped (and flagged once).
__device__ __forceinline__ void warp_histogram(const int32_t* idx, int c0, int c1, int E, int* wh_row, int lane,
                                               bool flag) {
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int b = c0; b < c1; b += 32) {
        const int f = b + lane;
        int e = (f < c1) ? idx[f] : -1;
        if (f < c1 && (e < 0 || e >= E)) {
            if (flag) atomicOr(&g_error_word, kErrBadExpert);
            e = -1;
        }
        const unsigned peers = same_expert_lanes(e, 32 - __clz(E));
        if (e >= 0 && (peers & lt_mask) == 0) wh_row[e] += __popc(peers);
    }
}

// Per expert, exclusive scan of the 32 warps' counts in place (warp ww scans
// experts ww, ww + 32, ..., lane = source warp); totals to cnt (if not null).
__device__ __forceinline__ void scan_over_warps(DispatchSmem& sm, int* cnt, int E, int warp, int lane) {
    for (int e = warp; e < E; e += kW) {
        const int v = sm.wh[lane][e];
        int inc = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += u;
        }
        sm.wh[lane][e] = inc - v;
        if (cnt && lane == 31) cnt[e] = inc;
    }
}

// From the per-expert totals in sm.cnt: offsets and token-tile bases (scan
// over experts by warp 0), then offsets, the tile list and (tile count, rows
// of the largest tile) to global memory. Every thread of the CTA calls it.
__device__ __forceinline__ void finish_experts(const DispatchArgs& a, DispatchSmem& sm, int tid, int warp,
                                               int lane, bool write_out = true) {
    const int E = a.E;
    if (warp == 0) {  // lane owns experts [8 lane, 8 lane + 8)
        int lc[8], lt[8], sc = 0, st = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int e = lane * 8 + j;
            lc[j] = (e < E) ? sm.cnt[e] : 0;
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
                sm.off[e] = rc;
                sm.tbase[e] = rt;
            }
            rc += lc[j];
            rt += lt[j];
        }
        if (lane == 31) {
            sm.off[E] = ic;
            sm.tbase[E] = it;
        }
    }
    __syncthreads();
    if (!write_out) return;
    for (int e = tid; e <= E; e += blockDim.x) a.offsets[e] = sm.off[e];
    if (a.tiles) {
        for (int e = tid; e < E; e += blockDim.x) {
            for (int i = 0; sm.tbase[e] + i < sm.tbase[e + 1]; ++i) {
                Tile t;
                t.e = e;
                t.p0 = sm.off[e] + i * a.nmax;
                t.rows = min(a.nmax, sm.cnt[e] - i * a.nmax);
                t.pad = 0;
                a.tiles[sm.tbase[e] + i] = t;
            }
        }
        if (warp == 0 && a.num_tiles) {
            int mx = 0;
            for (int e = lane; e < E; e += 32) mx = max(mx, min(sm.cnt[e], a.nmax));
            mx = __reduce_max_sync(0xffffffffu, mx);
            if (lane == 0) {
                a.num_tiles[0] = sm.tbase[E];
                a.num_tiles[1] = mx;
            }
        }
    }
}

// Stable scatter of the slots [c0, c1) in slot order: slot f with expert e
// goes to the warp's running base for e plus its rank among equal ids in its
// 32-slot group.
__device__ __forceinline__ void warp_scatter(const DispatchArgs& a, int c0, int c1, int* wh_row, int lane) {
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int b = c0; b < c1; b += 32) {
        const int f = b + lane;
        int e = (f < c1) ? a.idx[f] : -1;
        if (e >= a.E || e < 0) e = -1;
        const unsigned peers = same_expert_lanes(e, 32 - __clz(a.E));
        const int rank = __popc(peers & lt_mask);
        if (e >= 0) {
            const int p = wh_row[e] + rank;
            a.perm[p] = f;
            a.inv[f] = p;
        } else if (f < c1) {
            a.inv[f] = -1;  // a dropped slot: the combine skips it
        }
        __syncwarp();
        if (e >= 0 && rank == 0) wh_row[e] += __popc(peers);
        __syncwarp();
    }
}

__device__ __forceinline__ void zero_warp_counts(DispatchSmem& sm, int tid) {
    for (int i = tid; i < kW * (kMaxE + 1); i += kDispatchThreads) (&sm.wh[0][0])[i] = 0;
}

// Slot chunk of CTA c in the three-kernel path.
__host__ __device__ inline int chunk_slots(int S) {
    const int c = (S + kDispatchMaxChunks - 1) / kDispatchMaxChunks;
    return max(2048, (c + 31) & ~31);
}
}  // namespace

// One CTA of 32 warps sorts everything; warp w owns the contiguous slot range
// [w*per, (w+1)*per). Warps cover the slots in order, so the sort is stable
// and the result unique. A lane keeps its (at most 8) expert ids in
// registers from one round of loads for both passes.
__global__ void __launch_bounds__(kDispatchThreads) dispatch_kernel(DispatchArgs a) {
    __shared__ DispatchSmem sm;
    constexpr int kPerLane = kDispatchSingleMaxSlots / kDispatchThreads;  // 8
    pdl_trigger();
    pdl_wait();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int per = (a.S + kW - 1) / kW;
    const int c0 = min(a.S, warp * per), c1 = min(a.S, c0 + per);
    int ev[kPerLane];
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
        const int f = c0 + 32 * i + lane;
        int e = (f < c1) ? a.idx[f] : -1;
        if (f < c1 && (e < 0 || e >= a.E)) {
            atomicOr(&g_error_word, kErrBadExpert);
            e = -1;
        }
        ev[i] = e;
    }
    zero_warp_counts(sm, tid);
    __syncthreads();
    const unsigned lt_mask = (1u << lane) - 1u;
    int* wh = sm.wh[warp];
    // the lanes with the same expert in each 32-slot group, found once and
    // used by both passes: by ballots when the warps' groups are full (the
    // match instruction is the costly one there: canvas histogram 2.1 -> 1.2
    // us), by the match when they hold a few ids (decode: 0.2 against 0.7 us)
    const bool full_groups = a.S >= 32 * kW;
    unsigned pm[kPerLane];
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
        pm[i] = 0u;
        if (c0 + 32 * i >= c1) break;  // warp-uniform
        pm[i] = full_groups ? same_expert_lanes(ev[i], 32 - __clz(a.E)) : __match_any_sync(0xffffffffu, ev[i]);
        if (ev[i] >= 0 && (pm[i] & lt_mask) == 0) wh[ev[i]] += __popc(pm[i]);
    }
    __syncthreads();
    scan_over_warps(sm, sm.cnt, a.E, warp, lane);
    __syncthreads();
    finish_experts(a, sm, tid, warp, lane);
    // the warp's own bases (the scatter reads no other warp's row)
    for (int e = lane; e < a.E; e += 32) wh[e] += sm.off[e];
    __syncwarp();
    // stable scatter in slot order from the warp's running bases
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
        if (c0 + 32 * i >= c1) break;  // warp-uniform
        const int f = c0 + 32 * i + lane, e = ev[i];
        const unsigned peers = pm[i];
        const int rank = __popc(peers & lt_mask);
        if (e >= 0) {
            const int p = wh[e] + rank;
            a.perm[p] = f;
            a.inv[f] = p;
        } else if (f < c1) {
            a.inv[f] = -1;  // a dropped slot: the combine skips it
        }
        __syncwarp();
        if (e >= 0 && rank == 0) wh[e] += __popc(peers);
        __syncwarp();
    }
}

// Dispatch fused with the gather (S <= kDispatchSingleMaxSlots): every CTA
// redoes the whole counting sort in shared memory (2 K slots: cheap, and no
// CTA waits for another), then writes the sorted rows [r0, r0 + rows) of its
// own range: perm, inv and xs[p] = interleave(x[perm[p] / k]). CTA 0 also
// writes the offsets and the tile list. The result equals dispatch_kernel's
// followed by gather_kernel's.
__global__ void __launch_bounds__(kDispatchThreads) dispatch_gather_kernel(DispatchArgs a,
                                                                           const uint16_t* __restrict__ x,
                                                                           uint16_t* __restrict__ xs, int k, int H,
                                                                           int rows) {
    __shared__ DispatchSmem sm;
    __shared__ int32_t src_tok[kFusedMaxRows];  // token of each row of this CTA's range
    constexpr int kPerLane = kDispatchSingleMaxSlots / kDispatchThreads;  // 8
    pdl_trigger();
    pdl_wait();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r0 = blockIdx.x * rows, r1 = r0 + rows;
    const int per = (a.S + kW - 1) / kW;
    const int c0 = min(a.S, warp * per), c1 = min(a.S, c0 + per);
    int ev[kPerLane];
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
        const int f = c0 + 32 * i + lane;
        int e = (f < c1) ? a.idx[f] : -1;
        if (f < c1 && (e < 0 || e >= a.E)) {
            if (blockIdx.x == 0) atomicOr(&g_error_word, kErrBadExpert);
            e = -1;
        }
        ev[i] = e;
    }
    zero_warp_counts(sm, tid);
    for (int i = tid; i < rows; i += kDispatchThreads) src_tok[i] = -1;
    __syncthreads();
    const unsigned lt_mask = (1u << lane) - 1u;
    int* wh = sm.wh[warp];
    // the lanes with the same expert in each 32-slot group, found once and
    // used by both passes: by ballots when the warps' groups are full (the
    // match instruction is the costly one there: canvas histogram 2.1 -> 1.2
    // us), by the match when they hold a few ids (decode: 0.2 against 0.7 us)
    const bool full_groups = a.S >= 32 * kW;
    unsigned pm[kPerLane];
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
        pm[i] = 0u;
        if (c0 + 32 * i >= c1) break;  // warp-uniform
        pm[i] = full_groups ? same_expert_lanes(ev[i], 32 - __clz(a.E)) : __match_any_sync(0xffffffffu, ev[i]);
        if (ev[i] >= 0 && (pm[i] & lt_mask) == 0) wh[ev[i]] += __popc(pm[i]);
    }
    __syncthreads();
    scan_over_warps(sm, sm.cnt, a.E, warp, lane);
    __syncthreads();
    finish_experts(a, sm, tid, warp, lane, blockIdx.x == 0);
    // the warp's own bases (the scatter reads no other warp's row)
    for (int e = lane; e < a.E; e += 32) wh[e] += sm.off[e];
    __syncwarp();
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
        if (c0 + 32 * i >= c1) break;  // warp-uniform
        const int f = c0 + 32 * i + lane, e = ev[i];
        const unsigned peers = pm[i];
        const int rank = __popc(peers & lt_mask);
        if (e >= 0) {
            const int p = wh[e] + rank;
            if (p >= r0 && p < r1) {
                a.perm[p] = f;
                a.inv[f] = p;
                src_tok[p - r0] = f / k;
            }
        } else if (f < c1 && blockIdx.x == 0) {
            a.inv[f] = -1;  // a dropped slot: the combine skips it
        }
        __syncwarp();
        if (e >= 0 && rank == 0) wh[e] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    // One warp a row: 16-byte chunks of x[t], interleaved, lane-strided.
    const int chunks = H / 8;
    for (int rr = warp; rr < rows; rr += kW) {
        const int t = src_tok[rr];
        if (t < 0) continue;  // past the last valid slot
        const uint4* srow = reinterpret_cast<const uint4*>(x + (size_t)t * H);
        uint4* drow = reinterpret_cast<uint4*>(xs + (size_t)(r0 + rr) * H);
#pragma unroll 4
        for (int c = lane; c < chunks; c += 32) drow[c] = interleave8(__ldg(srow + c));
    }
}

// Three-kernel path for large S. 1: CTA c counts its slot chunk by expert.
__global__ void __launch_bounds__(kDispatchThreads) dispatch_count_kernel(DispatchArgs a) {
    __shared__ DispatchSmem sm;
    pdl_trigger();
    pdl_wait();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int chunk = chunk_slots(a.S);
    const int s0 = blockIdx.x * chunk, s1 = min(a.S, s0 + chunk);
    zero_warp_counts(sm, tid);
    __syncthreads();
    const int per = (s1 - s0 + kW - 1) / kW;
    const int c0 = min(s1, s0 + warp * per), c1 = min(s1, c0 + per);
    warp_histogram(a.idx, c0, c1, a.E, sm.wh[warp], lane, true);
    __syncthreads();
    for (int e = tid; e < a.E; e += kDispatchThreads) {
        int t = 0;
        for (int w = 0; w < kW; ++w) t += sm.wh[w][e];
        a.chunk_hist[blockIdx.x * a.E + e] = t;
    }
}

// 2: one CTA: per-expert totals and chunk prefixes, offsets, tiles; the
// chunk histogram becomes each chunk's base position per expert. G adjacent
// threads share an expert, each loading a run of consecutive chunks at once,
// then a scan over the G runs by shuffles, and each writes its chunks'
// final bases once (offset included).
__global__ void __launch_bounds__(kDispatchThreads) dispatch_scan_kernel(DispatchArgs a) {
    __shared__ DispatchSmem sm;
    constexpr int kMaxRun = (kDispatchMaxChunks + 3) / 4;  // chunks a thread (G >= 4)
    static_assert(kDispatchThreads / 4 >= kMaxE, "G >= 4 threads an expert");
    pdl_trigger();
    pdl_wait();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nch = (a.S + chunk_slots(a.S) - 1) / chunk_slots(a.S);  // <= kDispatchMaxChunks
    const int G = a.E <= kDispatchThreads / 8 ? 8 : 4;                 // threads an expert (divides 32)
    const int e = tid / G, m = tid % G;
    const int run = (nch + G - 1) / G;  // <= kMaxRun
    const int cb = m * run;             // this thread's first chunk
    int v[kMaxRun];
    int sum = 0;
#pragma unroll
    for (int j = 0; j < kMaxRun; ++j) {
        v[j] = (e < a.E && j < run && cb + j < nch) ? a.chunk_hist[(cb + j) * a.E + e] : 0;
        sum += v[j];
    }
    // inclusive scan of the runs' sums over the expert's G threads
    int inc = sum;
    for (int o = 1; o < G; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, inc, o, G);
        if (m >= o) inc += u;
    }
    if (e < a.E && m == G - 1) sm.cnt[e] = inc;  // the expert's total
    __syncthreads();
    finish_experts(a, sm, tid, warp, lane);
    if (e < a.E) {
        int base = sm.off[e] + inc - sum;
#pragma unroll
        for (int j = 0; j < kMaxRun; ++j) {
            if (j < run && cb + j < nch) {
                a.chunk_hist[(cb + j) * a.E + e] = base;
                base += v[j];
            }
        }
    }
}

// 3: CTA c scatters its chunk from the chunk's per-expert bases.
__global__ void __launch_bounds__(kDispatchThreads) dispatch_scatter_kernel(DispatchArgs a) {
    __shared__ DispatchSmem sm;
    pdl_trigger();
    pdl_wait();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int chunk = chunk_slots(a.S);
    const int s0 = blockIdx.x * chunk, s1 = min(a.S, s0 + chunk);
    zero_warp_counts(sm, tid);
    __syncthreads();
    const int per = (s1 - s0 + kW - 1) / kW;
    const int c0 = min(s1, s0 + warp * per), c1 = min(s1, c0 + per);
    warp_histogram(a.idx, c0, c1, a.E, sm.wh[warp], lane, false);
    __syncthreads();
    scan_over_warps(sm, nullptr, a.E, warp, lane);
    __syncthreads();
    for (int i = tid; i < kW * a.E; i += kDispatchThreads)
        sm.wh[i / a.E][i % a.E] += a.chunk_hist[blockIdx.x * a.E + i % a.E];
    __syncthreads();
    warp_scatter(a, c0, c1, sm.wh[warp], lane);
}

cudaError_t launch_dispatch_gather(const DispatchArgs& a, const uint16_t* x, uint16_t* xs, int k, int H, int sms,
                                   cudaStream_t stream) {
    if (a.S == 0) return cudaSuccess;
    // One wave (a 1024-thread CTA of 64 registers fills an SM): at least 8
    // rows (45 KB at H = 2816) a CTA, at most one CTA an SM.
    const int rows = std::max(8, (a.S + sms - 1) / std::max(1, sms));
    if (a.S > kDispatchSingleMaxSlots || rows > kFusedMaxRows) return cudaErrorInvalidValue;
    const int grid = (a.S + rows - 1) / rows;
    return launch_pdl(dispatch_gather_kernel, dim3(grid), dim3(kDispatchThreads), 0, stream, a, x, xs, k, H, rows);
}

cudaError_t launch_dispatch(const DispatchArgs& a, cudaStream_t stream) {
    if (a.S <= kDispatchSingleMaxSlots)  // the one-CTA sort holds up to 8 slots a thread in registers
        return launch_pdl(dispatch_kernel, dim3(1), dim3(kDispatchThreads), 0, stream, a);
    if (a.chunk_hist == nullptr) return cudaErrorInvalidValue;
    const int nch = (a.S + chunk_slots(a.S) - 1) / chunk_slots(a.S);  // <= kDispatchMaxChunks
    cudaError_t e = launch_pdl(dispatch_count_kernel, dim3(nch), dim3(kDispatchThreads), 0, stream, a);
    if (e == cudaSuccess) e = launch_pdl(dispatch_scan_kernel, dim3(1), dim3(kDispatchThreads), 0, stream, a);
    if (e == cudaSuccess) e = launch_pdl(dispatch_scatter_kernel, dim3(nch), dim3(kDispatchThreads), 0, stream, a);
    return e;
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
// out[t] = bf16(sum_j bf16(y_j * w[t k + j])), y_j = row inv[t k + j] of the
// down product (stored by sorted row), the products rounded to bf16 (the
// product of two bf16 arrays is a bf16 array) and summed in fp32 in j order.
// fp32 sums, in slot order j, of bf16(y[inv[j]] * w[j]) over the 8 elements
// of one 16-byte chunk (yc: the chunk in row 0 of y; rows are `chunks`
// chunks apart). For k <= 8 every row's load is issued before the sums, so
// the k reads are in flight together (the combine measured ~10% faster at
// T = 256 and T = 4096 than with one row a step); dropped slots (inv < 0)
// add nothing.
__device__ __forceinline__ void combine_chunk(const uint4* __restrict__ yc, int chunks, const int32_t* __restrict__ it,
                                              const uint16_t* __restrict__ wt, int k, float (&acc)[8]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    auto add = [&](const uint4& v, uint32_t wb) {
        const uint32_t w2 = wb | (wb << 16);
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint32_t pr = mul_bf16x2(u[q], w2);  // bf16(y * w), both halves
            acc[2 * q] = __fadd_rn(acc[2 * q], __uint_as_float(pr << 16));
            acc[2 * q + 1] = __fadd_rn(acc[2 * q + 1], __uint_as_float(pr & 0xFFFF0000u));
        }
    };
    if (k <= 8) {
        int p[8];
        uint32_t wv[8];
        uint4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            p[j] = j < k ? __ldg(it + j) : -1;
            wv[j] = j < k ? (uint32_t)__ldg(wt + j) : 0u;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = p[j] >= 0 ? __ldg(yc + (size_t)p[j] * chunks) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (p[j] >= 0) add(v[j], wv[j]);
    } else {
        for (int j = 0; j < k; ++j) {
            const int p = __ldg(it + j);
            if (p < 0) continue;  // slot dropped by the dispatch (expert id out of range)
            add(__ldg(yc + (size_t)p * chunks), __ldg(wt + j));
        }
    }
}

__global__ void __launch_bounds__(128) combine_kernel(const uint16_t* __restrict__ y,
                                                      const int32_t* __restrict__ inv,
                                                      const uint16_t* __restrict__ w,
                                                      uint16_t* __restrict__ out, int k, int H) {
    pdl_trigger();
    pdl_wait();
    const int chunks = H / 8;
    const int t = blockIdx.x, c = blockIdx.y * 128 + threadIdx.x;
    if (c >= chunks) return;
    float acc[8];
    combine_chunk(reinterpret_cast<const uint4*>(y) + c, chunks, inv + (size_t)t * k, w + (size_t)t * k, k, acc);
    reinterpret_cast<uint4*>(out + (size_t)t * H)[c] =
        make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                   pack_bf16x2(acc[6], acc[7]));
}

// Combine followed by the MoE branch's post norm (postFfNorm2), one CTA a
// token: c = the combined row (bf16, as combine_kernel), then
// out = bf16((c * rsqrt(mean(c^2) + eps)) * post_w) with fp32 steps; the sum of
// squares is carried as an error-free two-float sum, so the fp32 mean is the
// exact mean rounded once (unless within ~2^-40 of a rounding boundary).
constexpr int kNormThreads = 256;
constexpr int kNormChunks = 4;  // 16-byte chunks a thread: H <= 8192
__global__ void __launch_bounds__(kNormThreads) combine_norm_kernel(const uint16_t* __restrict__ y,
                                                                    const int32_t* __restrict__ inv,
                                                                    const uint16_t* __restrict__ w,
                                                                    const uint16_t* __restrict__ post_w,
                                                                    uint16_t* __restrict__ out, int k, int H,
                                                                    float eps) {
    pdl_trigger();
    pdl_wait();
    const int chunks = H / 8, t = blockIdx.x, tid = threadIdx.x;
    const uint4* y4 = reinterpret_cast<const uint4*>(y);
    const uint16_t* wt = w + (size_t)t * k;
    const int32_t* it = inv + (size_t)t * k;
    uint4 cv[kNormChunks];
    float hi = 0.f, lo = 0.f;
#pragma unroll
    for (int q = 0; q < kNormChunks; ++q) {
        const int c = tid + q * kNormThreads;
        cv[q] = make_uint4(0, 0, 0, 0);
        if (c >= chunks) continue;
        float acc[8];
        combine_chunk(y4 + c, chunks, it, wt, k, acc);
        const uint32_t b0 = pack_bf16x2(acc[0], acc[1]), b1 = pack_bf16x2(acc[2], acc[3]),
                       b2 = pack_bf16x2(acc[4], acc[5]), b3 = pack_bf16x2(acc[6], acc[7]);
        cv[q] = make_uint4(b0, b1, b2, b3);
        sumsq_bf16x2(b0, hi, lo);
        sumsq_bf16x2(b1, hi, lo);
        sumsq_bf16x2(b2, hi, lo);
        sumsq_bf16x2(b3, hi, lo);
    }
    const float rs = block_rsqrt_mean<kNormThreads>(hi, lo, H, eps);
#pragma unroll
    for (int q = 0; q < kNormChunks; ++q) {
        const int c = tid + q * kNormThreads;
        if (c >= chunks) continue;
        const uint4 pw = __ldg(reinterpret_cast<const uint4*>(post_w) + c);
        const uint32_t xv[4] = {cv[q].x, cv[q].y, cv[q].z, cv[q].w}, wv[4] = {pw.x, pw.y, pw.z, pw.w};
        uint32_t o4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
            o4[e] = pack_bf16x2(
                __fmul_rn(__fmul_rn(__uint_as_float(xv[e] << 16), rs), __uint_as_float(wv[e] << 16)),
                __fmul_rn(__fmul_rn(__uint_as_float(xv[e] & 0xFFFF0000u), rs), __uint_as_float(wv[e] & 0xFFFF0000u)));
        reinterpret_cast<uint4*>(out + (size_t)t * H)[c] = make_uint4(o4[0], o4[1], o4[2], o4[3]);
    }
}

cudaError_t launch_combine_norm(const uint16_t* y, const int32_t* inv, const uint16_t* w, const uint16_t* post_w,
                                uint16_t* out, int T, int k, int H, float eps, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    if (H / 8 > kNormThreads * kNormChunks) return cudaErrorInvalidValue;
    return launch_pdl(combine_norm_kernel, dim3((unsigned)T), dim3(kNormThreads), 0, stream, y, inv, w, post_w, out,
                      k, H, eps);
}

cudaError_t launch_combine(const uint16_t* y, const int32_t* inv, const uint16_t* w, uint16_t* out, int T, int k,
                           int H, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const dim3 grid((unsigned)T, (unsigned)((H / 8 + 127) / 128));
    return launch_pdl(combine_kernel, grid, dim3(128), 0, stream, y, inv, w, out, k, H);
}

// dst[i] = src[i] for `bytes` bytes (a multiple of 16, both 16-byte
// aligned), grid-stride, 16 bytes a thread a step. src may be pinned host
// memory mapped into the device's address space: the copy then reads it
// over the host link from every SM at once.
__global__ void __launch_bounds__(256) copy16_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src,
                                                     size_t n) {
    pdl_trigger();
    pdl_wait();
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        dst[i] = src[i];
}

cudaError_t launch_copy16(void* dst, const void* src, size_t bytes, int sms, cudaStream_t stream) {
    if (bytes == 0) return cudaSuccess;
    if (bytes % 16 != 0) return cudaErrorInvalidValue;
    const size_t n = bytes / 16;
    const size_t blocks = (n + 255) / 256;
    const unsigned grid = (unsigned)(blocks < (size_t)sms * 4 ? blocks : (size_t)sms * 4);
    return launch_pdl(copy16_kernel, dim3(grid), dim3(256), 0, stream, static_cast<uint4*>(dst),
                      static_cast<const uint4*>(src), n);
}

int dispatch_error_word() {
    int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_error_word, sizeof(int)) != cudaSuccess) return 0;
    cudaMemcpyToSymbol(g_error_word, &z, sizeof(int));
    return v;
}

}  // namespace moe
