// Small-token dequant-GEMV for the two QuantizedSwitchLinear calls of
// DiffExperts.forward ("diffusion-gemma/model.ts"), gate_up with the split +
// GeGLU fused into its epilogue, and down: the regime of a few rows per
// expert (a decode step: T = 8 tokens, about 52 experts with one or two rows
// each), where the tensor cores would multiply mostly padding and the work
// is streaming the packed weights from HBM.
//
// Each weight is dequantised exactly as the grouped GEMM does it, w =
// bf16(S q + B) (four nibble pairs of a packed word become bf16 pairs with
// one lop3, the exact q with one bf16x2 fma, and S q + B rounded once with
// another), and each product x w is a mixed bf16 x bf16 -> fp32 fma on
// register halves, accumulated in fp32 along K. The results equal the
// grouped GEMM's up to the order of the fp32 sums.
//
// Persistent, one CTA per SM, work item = (token tile of up to 4 rows of
// one expert, 128-row weight tile), K in stages of 256:
//   warp 0     TMA producer: the packed-weight ring (128 rows x 128 B a stage,
//              128-byte swizzle, as the grouped GEMM), and per item the
//              group scales and biases and the item's token rows (bulk
//              copies, double-buffered);
//   warps 1-16 the dot products: warp w takes 8 weight rows, lane (kq, rr)
//              row rr and the 64-wide quarter kq of each stage's K (for
//              gate_up the 8 rows are 4 gate rows and the 4 up rows of the
//              same outputs, so the GeGLU pairs sit in lanes l, l ^ 4); the
//              lanes of a K quarter read the same token chunk, a shared
//              memory broadcast. Each token's sum runs as four independent
//              fp32 chains (one per nibble pair), added in a fixed order.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kStageK = 256;
constexpr int kPackedStageBytes = 128 * 128;  // 128 rows x 32 words
constexpr int kMaxStages = 8;
constexpr int kComputeWarps = 16;
constexpr int kThreads = (1 + kComputeWarps) * 32;
constexpr uint32_t kSleepRing = 200;  // ns between tests of the producer's waits

struct GvSmem {
    uint64_t wfull[kMaxStages], wempty[kMaxStages];  // packed-weight ring
    uint64_t sfull[2], sempty[2];                    // scales + biases of an item
    uint64_t xfull[2], xempty[2];                    // token rows of an item
    int abort_flag;
};

__host__ __device__ inline int gv_scale_bytes(int K) { return ((128 * (K / 64) * 2 * 2) + 1023) & ~1023; }
__host__ __device__ inline int gv_x_bytes(int K) { return (kGemvRows * K * 2 + 1023) & ~1023; }

// fp32 d = a * b + c for bf16 a, b given as 16-bit halves of 32-bit registers.
__device__ __forceinline__ float fma_bf16_lo(uint32_t a, uint32_t b, float c) {
    float d;
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, al, bl, %3;\n\t}"
        : "=f"(d)
        : "r"(a), "r"(b), "f"(c));
    return d;
}
__device__ __forceinline__ float fma_bf16_hi(uint32_t a, uint32_t b, float c) {
    float d;
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, ah, bh, %3;\n\t}"
        : "=f"(d)
        : "r"(a), "r"(b), "f"(c));
    return d;
}

}  // namespace

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    gemv_kernel(const __grid_constant__ CUtensorMap wmap, GemmArgs a, const uint16_t* __restrict__ xsrc) {
    extern __shared__ __align__(1024) uint8_t dsmem[];
    __shared__ GvSmem sh;
    pdl_trigger();
    // Warm L2 with the weights and scales of this CTA's first items before
    // waiting for the routing (as the grouped GEMM; only data no earlier
    // kernel writes).
    if (threadIdx.x == 0 && a.prefetch_items > 0) {
        const uint32_t row_bytes = (uint32_t)a.K / 2, G = (uint32_t)a.K / 64;
        for (int i = 0; i < a.prefetch_items; ++i) {
            const int it = blockIdx.x + i * gridDim.x;
            const int ti = it / a.n_tiles, j = it % a.n_tiles;
            const int e = ti / a.tiles_per_expert;
            if (e >= a.E) break;
            for (int h = 0; h < (MODE == kGateUp ? 2 : 1); ++h) {
                const size_t r0 = (MODE == kGateUp) ? (size_t)e * a.N + (size_t)h * a.inter + 64 * j
                                                    : (size_t)e * a.N + 128 * j;
                const uint32_t rows = (MODE == kGateUp) ? 64u : 128u;
                prefetch_l2_bulk(a.w + r0 * row_bytes, rows * row_bytes);
                prefetch_l2_bulk(a.scales + r0 * G, (rows * G * 2 + 15) & ~15u);
                prefetch_l2_bulk(a.biases + r0 * G, (rows * G * 2 + 15) & ~15u);
            }
        }
    }
    pdl_wait();
    // 1024-byte aligned carve-up: packed ring | 2 scale buffers | 2 token buffers
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsmem) + 1023) & ~uintptr_t(1023));
    const int NP = a.wstages;
    const int K = a.K, G = K / 64;
    const int sbuf_bytes = gv_scale_bytes(K), xbuf_bytes = gv_x_bytes(K);
    uint8_t* wring = base;
    uint8_t* scale_base = wring + (size_t)NP * kPackedStageBytes;
    uint8_t* xbase = scale_base + 2 * (size_t)sbuf_bytes;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int* abort_flag = &sh.abort_flag;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NP; ++s) {
            mbar_init(&sh.wfull[s], 1);
            mbar_init(&sh.wempty[s], kComputeWarps);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sh.sfull[i], 1);
            mbar_init(&sh.sempty[i], kComputeWarps);
            mbar_init(&sh.xfull[i], 1);
            mbar_init(&sh.xempty[i], kComputeWarps);
        }
        sh.abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    const int ntok = a.num_tiles[0];
    const int num_items = ntok * a.n_tiles;
    const int nstages = (K + kStageK - 1) / kStageK;
    if (warp == 0) {
        // ------------------------------- weights, scales, token rows --
        if (elect_one()) prefetch_tensormap(&wmap);
        int slot = 0;
        uint32_t ph = 0, issued = 0;
        int li = 0;
        bool ok = true;
        for (int it = blockIdx.x; it < num_items && ok; it += gridDim.x, ++li) {
            const int ti = it / a.n_tiles, j = it % a.n_tiles;
            const Tile tl = a.tiles[ti];
            const int sb = li & 1;
            if (!(ok = mbar_wait(&sh.sempty[sb], ((li >> 1) & 1) ^ 1, abort_flag, kSleepRing, 1))) break;
            if (!(ok = mbar_wait(&sh.xempty[sb], ((li >> 1) & 1) ^ 1, abort_flag, kSleepRing, 4))) break;
            uint8_t* sbuf = scale_base + sb * sbuf_bytes;
            const uint32_t half = (uint32_t)(64 * G * 2);  // bytes of 64 rows
            const uint32_t xbytes = (uint32_t)tl.rows * (uint32_t)K * 2u;
            if (elect_one()) {
                mbar_arrive_expect_tx(&sh.sfull[sb], 4 * half);
                if (MODE == kGateUp) {
                    const size_t r_gate = (size_t)tl.e * a.N + 64 * j;
                    const size_t r_up = (size_t)tl.e * a.N + a.inter + 64 * j;
                    bulk_load(sbuf, a.scales + r_gate * G, half, &sh.sfull[sb]);
                    bulk_load(sbuf + half, a.scales + r_up * G, half, &sh.sfull[sb]);
                    bulk_load(sbuf + 2 * half, a.biases + r_gate * G, half, &sh.sfull[sb]);
                    bulk_load(sbuf + 3 * half, a.biases + r_up * G, half, &sh.sfull[sb]);
                } else {
                    const size_t r0 = (size_t)tl.e * a.N + 128 * j;
                    bulk_load(sbuf, a.scales + r0 * G, 2 * half, &sh.sfull[sb]);
                    bulk_load(sbuf + 2 * half, a.biases + r0 * G, 2 * half, &sh.sfull[sb]);
                }
                // the item's token rows p0 .. p0 + rows - 1 (contiguous, K-interleaved)
                mbar_arrive_expect_tx(&sh.xfull[sb], xbytes);
                bulk_load(xbase + sb * xbuf_bytes, xsrc + (size_t)tl.p0 * K, xbytes, &sh.xfull[sb]);
            }
            __syncwarp();
            for (int s = 0; s < nstages; ++s) {
                if (!(ok = mbar_wait(&sh.wempty[slot], ph ^ 1, abort_flag, kSleepRing, 2))) break;
                uint8_t* st = wring + (size_t)slot * kPackedStageBytes;
                if (elect_one()) {
                    mbar_arrive_expect_tx(&sh.wfull[slot], kPackedStageBytes);
                    if (MODE == kGateUp) {
                        tma_load_2d(st, &wmap, &sh.wfull[slot], s * 32, tl.e * a.N + 64 * j);
                        tma_load_2d(st + 64 * 128, &wmap, &sh.wfull[slot], s * 32, tl.e * a.N + a.inter + 64 * j);
                    } else {
                        tma_load_2d(st, &wmap, &sh.wfull[slot], s * 32, tl.e * a.N + 128 * j);
                    }
                }
                __syncwarp();
                ++issued;
                if (++slot == NP) {
                    slot = 0;
                    ph ^= 1;
                }
            }
        }
        // Do not leave while copies into shared memory are in flight.
        for (uint32_t g = (issued > (uint32_t)NP ? issued - NP : 0); g < issued; ++g)
            mbar_drain(&sh.wfull[g % NP], (g / NP) & 1);
        for (int l = (li > 2 ? li - 2 : 0); l < li; ++l) {
            mbar_drain(&sh.sfull[l & 1], (l >> 1) & 1);
            mbar_drain(&sh.xfull[l & 1], (l >> 1) & 1);
        }
    } else {
        // ------------------------------------------------ dot products --
        const int cw = warp - 1;       // 0..15
        const int kq = lane >> 3;      // which 64-wide quarter (atom) of a stage's K
        const int rr = lane & 7;
        int row;                       // row of the weight stage (and of the scale buffer)
        if (MODE == kGateUp)
            row = (rr < 4) ? (4 * cw + rr) : (64 + 4 * cw + (rr - 4));
        else
            row = 8 * cw + rr;
        // this thread's two 16-byte chunks (its atom) of its row in ring slot 0 (swizzled)
        const uint32_t wo0 = smem_u32(wring) + (uint32_t)row * 128u + ((uint32_t)((2 * kq) ^ (row & 7)) << 4);
        const uint32_t wo1 = smem_u32(wring) + (uint32_t)row * 128u + ((uint32_t)((2 * kq + 1) ^ (row & 7)) << 4);
        const uint32_t srow = smem_u32(scale_base) + (uint32_t)(row * G) * 2u;
        const uint32_t bias_off = (uint32_t)(128 * G * 2);
        int wslot = 0;
        uint32_t wph = 0;
        bool ok = true;
        int li = 0;
        for (int it = blockIdx.x; it < num_items && ok; it += gridDim.x, ++li) {
            const int ti = it / a.n_tiles, j = it % a.n_tiles;
            const Tile tl = a.tiles[ti];
            const int rows = tl.rows;
            const int sb = li & 1;
            if (!(ok = mbar_wait(&sh.sfull[sb], (li >> 1) & 1, abort_flag, 0, 8))) break;
            if (!(ok = mbar_wait(&sh.xfull[sb], (li >> 1) & 1, abort_flag, 0, 13))) break;
            const uint32_t sS = srow + (uint32_t)(sb * sbuf_bytes);
            const uint32_t xs = smem_u32(xbase + sb * xbuf_bytes);
            float acc[kGemvRows][4];
#pragma unroll
            for (int t = 0; t < kGemvRows; ++t)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[t][c] = 0.f;
            for (int s = 0; s < nstages; ++s) {
                const int atoms = min(kStageK, K - s * kStageK) / 64;  // 1..4
                if (!(ok = mbar_wait(&sh.wfull[wslot], wph, abort_flag, 0, 9))) break;
                if (kq < atoms) {  // quarter-uniform
                    const uint32_t so = (uint32_t)(wslot * kPackedStageBytes);
                    const int g = s * 4 + kq;
                    const uint4 c0 = lds128(wo0 + so), c1 = lds128(wo1 + so);
                    uint32_t r[32];  // the atom's 64 weights, bf16(S q + B), pair c of word i at 4i + c
                    dequant_atom(c0, c1, lds_u16(sS + (uint32_t)(2 * g)), lds_u16(sS + bias_off + (uint32_t)(2 * g)), r);
#pragma unroll
                    for (int w8 = 0; w8 < 8; ++w8) {
                        const uint32_t koff = (uint32_t)((g * 64 + w8 * 8) * 2);
#pragma unroll
                        for (int t = 0; t < kGemvRows; ++t) {
                            if (t < rows) {  // warp-uniform
                                // token chunk of the same 8 K, in the same pair order
                                const uint4 x = lds128(xs + (uint32_t)(t * K * 2) + koff);
                                const uint32_t xv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                                for (int c = 0; c < 4; ++c) {
                                    acc[t][c] = fma_bf16_lo(r[4 * w8 + c], xv[c], acc[t][c]);
                                    acc[t][c] = fma_bf16_hi(r[4 * w8 + c], xv[c], acc[t][c]);
                                }
                            }
                        }
                    }
                }
                // The arrive releases the loads above: the slot may be refilled.
                __syncwarp();
                mbar_arrive_lane0(&sh.wempty[wslot]);
                if (++wslot == NP) {
                    wslot = 0;
                    wph ^= 1;
                }
            }
            if (!ok) break;
            // the item's scales and token rows are no longer read
            __syncwarp();
            mbar_arrive_lane0(&sh.sempty[sb]);
            mbar_arrive_lane0(&sh.xempty[sb]);
            // the four chains, then the four K quarters (lanes l ^ 8, l ^ 16), in a fixed order
            float y[kGemvRows];
#pragma unroll
            for (int t = 0; t < kGemvRows; ++t) {
                float v = __fadd_rn(__fadd_rn(acc[t][0], acc[t][1]), __fadd_rn(acc[t][2], acc[t][3]));
                v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 8));
                y[t] = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 16));
            }
            if (MODE == kGateUp) {
                // lanes 0-3: gate rows 64 j + 4 cw + l; lanes 4-7: the up rows of the same outputs
                const int n = 64 * j + 4 * cw + (rr & 3);
                const int pos = interleaved_pos(n);
#pragma unroll
                for (int t = 0; t < kGemvRows; ++t) {
                    const float up = __shfl_xor_sync(0xffffffffu, y[t], 4);
                    if (t < rows && lane < 4) {
                        const float gb = bf16_bits_to_f32(f32_to_bf16_bits(y[t]));  // z is a bf16 tensor
                        const float ub = bf16_bits_to_f32(f32_to_bf16_bits(up));
                        a.out[(size_t)(tl.p0 + t) * a.out_ld + pos] = (uint16_t)geglu_bf16(gb, ub);
                    }
                }
            } else {
                const int hrow = 128 * j + 8 * cw + rr;
#pragma unroll
                for (int t = 0; t < kGemvRows; ++t)
                    if (t < rows && lane < 8)
                        a.out[(size_t)(tl.p0 + t) * a.out_ld + hrow] = (uint16_t)f32_to_bf16_bits(y[t]);
            }
        }
    }
    __syncwarp();
    __syncthreads();
}

size_t gemv_smem_bytes(int K, int wstages) {
    return 1024 /* alignment slack */ + (size_t)wstages * kPackedStageBytes + 2 * (size_t)gv_scale_bytes(K) +
           2 * (size_t)gv_x_bytes(K);
}

int gemv_stages(int K) {
    const size_t limit = 232448 - 2048;  // 227 KB per CTA minus the static part
    int nw = kMaxStages;
    while (nw > 2 && gemv_smem_bytes(K, nw) > limit) --nw;
    return gemv_smem_bytes(K, nw) <= limit ? nw : 0;
}

template <int MODE>
static cudaError_t launch_gv(const CUtensorMap& wmap, const GemmArgs& a, const uint16_t* xsrc, int grid,
                             size_t smem, cudaStream_t stream) {
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        cudaError_t err =
            cudaFuncSetAttribute(gemv_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448 - 2048);
        if (err != cudaSuccess) return err;
        attr_set[dev] = true;
    }
    return launch_pdl(gemv_kernel<MODE>, dim3(grid), dim3(kThreads), smem, stream, wmap, a, xsrc);
}

cudaError_t launch_gemv(int mode, const CUtensorMap& wmap, const GemmArgs& a, const uint16_t* xsrc, int grid,
                        cudaStream_t stream) {
    if (a.wstages < 2 || a.nmax != kGemvRows) return cudaErrorInvalidValue;
    const size_t smem = gemv_smem_bytes(a.K, a.wstages);
    switch (mode) {
        case kGateUp: return launch_gv<kGateUp>(wmap, a, xsrc, grid, smem, stream);
        case kDown: return launch_gv<kDown>(wmap, a, xsrc, grid, smem, stream);
        default: return cudaErrorInvalidValue;
    }
}

int gemv_error_word() {
    int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_error_word, sizeof(int)) != cudaSuccess) return 0;
    cudaMemcpyToSymbol(g_error_word, &z, sizeof(int));
    return v;
}

}  // namespace moe
