// Internal interface between the C-ABI host code (moe_api.cu) and the
// kernels. Not installed; the public interface is include/moe.h.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// Launch with programmatic stream serialization: the kernel may be scheduled
// while the previous kernel of the stream still runs; it calls pdl_wait()
// before it reads or writes global memory.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// Router: x [T,H] -> idx [T,k], w [T,k].
struct RouterArgs {
    const uint16_t* x;
    const uint16_t* router_w;
    const uint16_t* router_scale;
    const uint16_t* per_expert_scale;
    int32_t* idx;
    uint16_t* w;
    int T, H, E, k;
    float eps;
    float root;  // bf16(H^-0.5) as a float
    int tt;      // tokens per cluster (16, 32 or 64), from router_tokens_per_cluster
    // Optional (both or neither): the MoE branch's expert input
    // xe = bf16((x * rsqrt(mean(x^2) + eps)) * pre_w), fp32 steps, from the
    // same per-token rms the router computes.
    const uint16_t* pre_w;  // [H] bf16
    uint16_t* xe;           // [T, H] bf16
    // Optional: the projection as a 4-bit group-64 weight (the pages'
    // QuantizedLinear) instead of router_w; E <= 128. Each CTA dequantises
    // its slice once, w = bf16(S * q + B), into the layout the dense path
    // copies in.
    const uint32_t* rq_w;   // [E, H/8]
    const uint16_t* rq_s;   // [E, H/64]
    const uint16_t* rq_b;   // [E, H/64]
};
size_t router_smem_bytes(int H, int E, int tt);
int router_tokens_per_cluster(int T, int H, int E);
// wmap: router_w as bf16 [E rows, H], box {64, min(E, 128)}, 128B swizzle.
// xmap: x as bf16 [T rows, H], box {64, tt}, 128B swizzle.
cudaError_t launch_router(const CUtensorMap& wmap, const CUtensorMap& xmap, const RouterArgs& a,
                          cudaStream_t stream);
int router_error_word();
// Row router: the same results as launch_router, one CTA per 16 tokens over
// the whole hidden dimension (no cluster); dense router weight only, E <=
// 128, H a multiple of 64 whose 16-row tile fits in shared memory beside
// the router_scale and pre_w rows and a ring of at least 2 weight stages of
// two K blocks (H <= 4416). xmap: x as bf16 [T rows, H], box {64, 16}, 128B swizzle; wmap as
// for launch_router. a.tt is unused.
bool router_rows_fits(int H, int E, bool q4);
bool router_prefer_rows(int T, int H, int E);  // fits, and the clusters would walk two or more waves
size_t router_rows_smem_bytes(int H);
cudaError_t launch_router_rows(const CUtensorMap& wmap, const CUtensorMap& xmap, const RouterArgs& a,
                               cudaStream_t stream);

// A token tile of one expert: rows [p0, p0 + rows) of the expert-sorted slots.
struct Tile {
    int e, p0, rows, pad;
};

// Dispatch: stable counting sort of the flat slots by expert + tile list.
struct DispatchArgs {
    const int32_t* idx;  // [S]
    int32_t* perm;       // [S]
    int32_t* offsets;    // [E+1]
    int32_t* inv;        // [S]
    Tile* tiles;         // [max_tiles] (may be null)
    int32_t* num_tiles;  // [2]: tile count, rows of the largest tile (may be null)
    int S, E, nmax;      // nmax: rows per token tile
    // Scratch of kDispatchMaxChunks x E ints for the three-kernel path (large
    // S); null: one CTA does the whole sort.
    int32_t* chunk_hist = nullptr;
};
constexpr int kDispatchMaxChunks = 64;
constexpr int kDispatchSingleMaxSlots = 8192;  // above this the sort runs as three kernels
cudaError_t launch_dispatch(const DispatchArgs& a, cudaStream_t stream);
// Dispatch and gather in one launch (S <= kDispatchSingleMaxSlots): the same
// perm, inv, offsets, tiles and xs as launch_dispatch then launch_gather.
cudaError_t launch_dispatch_gather(const DispatchArgs& a, const uint16_t* x, uint16_t* xs, int k, int H, int sms,
                                   cudaStream_t stream);

// Gather: xs[p] = x[perm[p] / k] with each 8-element block of K stored in
// the order (0,4,1,5,2,6,3,7), the order the grouped GEMM's dequantised
// weights come out in.
cudaError_t launch_gather(const uint16_t* x, const int32_t* perm, const int32_t* offsets, uint16_t* xs,
                          int S, int k, int H, int E, cudaStream_t stream);

// Combine: out[t] = bf16(sum_j bf16(y[inv[t*k+j]] * w[t*k+j])), fp32 sum in
// j order; y by sorted row, inv the sorted row of each flat slot.
cudaError_t launch_combine(const uint16_t* y, const int32_t* inv, const uint16_t* w, uint16_t* out, int T, int k,
                           int H, cudaStream_t stream);
// Combine, then the MoE branch's post norm: out[t] = bf16((c * rsqrt(mean(c^2)
// + eps)) * post_w) of the combined bf16 row c (fp32 steps). H <= 8192.
cudaError_t launch_combine_norm(const uint16_t* y, const int32_t* inv, const uint16_t* w, const uint16_t* post_w,
                                uint16_t* out, int T, int k, int H, float eps, cudaStream_t stream);
int dispatch_error_word();
// dst = src, `bytes` a multiple of 16, both 16-byte aligned; src may be
// mapped pinned host memory.
cudaError_t launch_copy16(void* dst, const void* src, size_t bytes, int sms, cudaStream_t stream);

// Dense MLP input: xs[t] = row t of x, or RMSNorm(x, pre_w) with fp32 steps
// (pre_w non-null), each 8-element block of K interleaved as the gather's;
// and the tile list of one expert whose token tiles of nmax rows cover all
// T rows (num_tiles: count, rows of the largest). H <= 8192.
cudaError_t launch_dense_prep(const uint16_t* x, const uint16_t* pre_w, float eps, uint16_t* xs, Tile* tiles,
                              int32_t* num_tiles, int T, int H, int nmax, cudaStream_t stream);
// out[t] = bf16((c * rsqrt(mean(c^2) + eps)) [* w]) of c = s[t], or of
// c = bf16(embeds[t] + s[t]) (embeds non-null); w null: no weight. H <= 8192.
cudaError_t launch_add_norm(const uint16_t* embeds, const uint16_t* s, const uint16_t* w, float eps, uint16_t* out,
                            int T, int H, cudaStream_t stream);

// Grouped dequant-GEMM on tcgen05 (one expert per token tile).
// kHead: the tied head, as kDown but the epilogue writes row (p0 + token)
// of out_f32 directly (no permutation): softcap(bf16 logit) in fp32.
enum GemmMode { kGateUp = 0, kDown = 1, kHead = 2 };
struct GemmArgs {
    const uint16_t* scales;   // [E, N, K/64]
    const uint16_t* biases;   // [E, N, K/64]
    const Tile* tiles;
    const int32_t* num_tiles; // [0] tile count, [1] rows of the largest tile
    uint16_t* out;            // gate_up: mid [S, inter]; down: y [S, H]; both by sorted row
    int K;                    // reduction length (H or inter)
    int N;                    // rows of the weight (2*inter or H)
    int inter;                // gate_up: split point
    int out_ld;               // row length of out (inter or H)
    int E;                    // experts
    int nmax;                 // rows per token tile (64 or 128)
    int n_tiles;              // weight-row tiles per token tile
    int wstages;              // packed-weight ring depth (shared memory)
    int bregion;              // bytes of shared memory for the B-operand ring
    // L2 warm-up before the kernel waits for its producers: the packed
    // weights (w, [E*N rows, K/2 bytes]) and scales of each CTA's first
    // `prefetch_items` items, guessing that token tile t belongs to expert
    // t / tiles_per_expert (0 items: none). A wrong guess costs only
    // bandwidth that the preceding kernels leave idle.
    const uint8_t* w;
    int prefetch_items;
    int tiles_per_expert;
    // Item order. 0: token-tile-major (it = tile * n_tiles + j). 1 (one
    // expert, several token tiles): weight-tile-major (it = j * tiles +
    // tile), so the token tiles of a weight tile run together and share its
    // copy in L2 instead of streaming the weights once per token tile.
    int weight_major;
    // kHead: logits [rows, out_ld] fp32 and the final-logit softcap
    // (cap * tanh(x / cap) of the bf16 logit x; cap <= 0: x itself).
    float* out_f32;
    float softcap;
};
// Maps of the B operand (xs or mid, bf16 [S rows, K]), 128B swizzle:
//   m[i]  S rows of K/64 atoms of 64: dims {64, S, K/64}, byte strides
//         {2K, 128}, box {64, R, min(4, K/64)} for R = 16 << i. One copy
//         loads a stage's atoms of R token rows, atom after atom;
//   m2    [S rows, K] with box {64, 16}: one copy a 16-row, 64-wide block.
// The kernels for token tiles of up to 64 rows load 16-row blocks (m2),
// those for up to 128 rows one box of the smallest R that holds the tile
// (m[i]): each measured the faster for its tile sizes.
struct BMaps {
    CUtensorMap m[4];
    CUtensorMap m2;
};
// wmap: packed weights as uint32 [E*N rows, K/8], box {32, 64 or 128}, 128B swizzle.
// mode: the GemmMode (the down kernel also holds its epilogue's staging tiles).
size_t gemm_smem_bytes(int mode, int K, int wstages, int bregion);
void gemm_stages(int mode, int K, int nmax, int* wstages, int* bregion);
cudaError_t launch_gemm(int mode, const CUtensorMap& wmap, const BMaps& bmaps, const GemmArgs& a, int grid,
                        cudaStream_t stream);
int gemm_error_word();

// Small-token dequant-GEMV (a few rows per expert): the same work items as
// the grouped GEMM with token tiles of up to kGemvRows rows, the products
// taken group-factored in fp32 on the CUDA cores, x = xs (gate_up, GeGLU
// epilogue into mid) or mid (down, y by sorted row). a.w serves only the L2
// warm-up, a.bregion is unused; a.wstages from gemv_stages(K); a.nmax must
// be kGemvRows.
constexpr int kGemvRows = 4;
size_t gemv_smem_bytes(int K, int wstages);
int gemv_stages(int K);  // weight-ring depth that fits (0: K too large)
cudaError_t launch_gemv(int mode, const CUtensorMap& wmap, const GemmArgs& a, const uint16_t* xsrc, int grid,
                        cudaStream_t stream);
int gemv_error_word();

}  // namespace moe
