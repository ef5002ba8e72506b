// Grouped 4-bit dequant-GEMM on the 5th-generation tensor cores (tcgen05):
// the two QuantizedSwitchLinear calls of DiffExperts.forward
// ("diffusion-gemma/model.ts"), gate_up with the split + GeGLU fused into its
// epilogue, and down.
//
// The product is computed transposed (D^T = W . X^T) so the weight rows fill
// the 128-row M side of the MMA and the few tokens an expert receives fill
// the N side (16..128): at small token counts every weight byte is read from
// HBM once and the tensor cores stay far from busy.
//
// Persistent kernel, one CTA per SM, work item = (token tile of one expert,
// 128-row weight tile). Warp roles:
//   warp 0      TMA producer: packed weights (128 rows x 128 B per stage,
//               128 B swizzle) and the token tile of the B operand; the
//               item's scales and biases by one bulk copy per block of rows.
//   warp 1      TMEM owner and MMA issuer (one thread).
//   warps 4-7   dequant: thread = weight row = TMEM lane. Reads 8 nibbles per
//               word from shared memory, makes exact bf16 codes with the
//               0x4300 magic (128+q) minus 128, then bf16(S*q + B) with one
//               fused multiply-add, and stores the row's 256-K slice into the
//               A-operand ring in tensor memory (tcgen05.st).
//   warps 8-11  epilogue: tcgen05.ld of the fp32 accumulator, bf16 rounding,
//               GeGLU (gate_up) or the scatter to flat slots (down).
// A stage is 256 of K. The dequantised pair order inside each 8-element block
// is (0,4),(1,5),(2,6),(3,7); the B operands (gathered x, GeGLU output) are
// stored in that same K order, so the MMA sums the same products.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kThreads = 384;
constexpr int kStageK = 256;
constexpr int kPackedStageBytes = 128 * 128;  // 128 rows x 32 words
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kPCol0 = 256;              // partial-sum regions at columns 256 and 384

struct Smem {
    uint64_t full[8], empty[8];
    uint64_t afull[2], aempty[2];
    uint64_t pfull[2], pempty[2];  // per-stage partial accumulators in TMEM
    uint64_t sfull[2], sempty[2];
    uint32_t tmem_base;
    int abort_flag;
};

__host__ __device__ constexpr int b_stage_bytes(int nmax) { return 4 * nmax * 128; }
__host__ __device__ constexpr int stage_bytes(int nmax) { return kPackedStageBytes + b_stage_bytes(nmax); }
__host__ __device__ inline int scale_buf_bytes(int K) {
    // scales + biases for 128 rows, rounded up to 1 KB
    return ((128 * (K / 64) * 2 * 2) + 1023) & ~1023;
}

// bf16(gelu_approx(g) * up) for bf16 g, up, where gelu_approx(g) =
// 0.5 g (1 + tanh(s)), s = sqrt(2/pi) (g + 0.044715 g^3). 0.5 (1 + tanh s) is
// the logistic of 2s, evaluated in that form so it keeps its relative
// accuracy where 1 + tanh(s) cancels (s << 0). p = g*up is exact in fp32.
// For s >= 0 the value is p - p*t with t = 1 - logistic(2s) > 0, formed by a
// fused multiply-add rounded toward zero: the exact value lies strictly
// between 0 and p, so an exact bf16 tie of p (large g, where t is below
// fp32's resolution of 1) rounds toward zero as the exact value does.
__device__ __forceinline__ uint32_t geglu_bf16(float g, float up) {
    const float c = 0.7978845608028654f;  // sqrt(2/pi)
    const float s = __fmul_rn(c, __fadd_rn(g, __fmul_rn(0.044715f, __fmul_rn(g, __fmul_rn(g, g)))));
    const float p = __fmul_rn(g, up);
    float m;
    if (s < 0.f) {
        const float e = expf(__fmul_rn(2.0f, s));
        m = __fmul_rn(p, __fdiv_rn(e, __fadd_rn(1.0f, e)));
    } else {
        const float e = expf(__fmul_rn(-2.0f, s));
        const float t = fmaxf(__fdiv_rn(e, __fadd_rn(1.0f, e)), 1e-30f);
        m = __fmaf_rz(-p, t, p);
    }
    return f32_to_bf16_bits(m);
}

// Position of element n inside its 8-block in the interleaved K order.
__device__ __forceinline__ int interleaved_pos(int n) {
    const int r = n & 7;
    return (n & ~7) | (r < 4 ? 2 * r : 2 * r - 7);
}

}  // namespace

template <int MODE, int NMAX>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap bmap,
                        GemmArgs a) {
    extern __shared__ __align__(1024) uint8_t dsmem[];
    __shared__ Smem sh;
    // 1024-byte aligned carve-up: [stages][packed | B atoms] then 2 scale buffers.
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsmem) + 1023) & ~uintptr_t(1023));
    const int NS = a.stages;
    const int sbytes = stage_bytes(NMAX);
    uint8_t* scale_base = base + (size_t)NS * sbytes;
    const int G = a.K / 64;  // groups per weight row
    const int sbuf_bytes = scale_buf_bytes(a.K);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int* abort_flag = &sh.abort_flag;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&sh.full[s], 1);
            mbar_init(&sh.empty[s], 5);  // 4 dequant warps + 1 MMA commit
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sh.afull[i], 128);
            mbar_init(&sh.aempty[i], 1);
            mbar_init(&sh.pfull[i], 1);
            mbar_init(&sh.pempty[i], 128);
            mbar_init(&sh.sfull[i], 1);
            mbar_init(&sh.sempty[i], 4);
        }
        sh.abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&wmap);
        prefetch_tensormap(&bmap);
    }
    if (warp == 1) {
        tmem_alloc(&sh.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;

    const int num_items = (*a.num_tiles) * a.n_tiles;
    const int K = a.K;
    const int nstages = (K + kStageK - 1) / kStageK;

    if (warp == 0) {
        // ------------------------------------------------------ producer --
        if (lane == 0) {
            uint32_t gs = 0;
            int li = 0;
            bool ok = true;
            for (int it = blockIdx.x; it < num_items && ok; it += gridDim.x, ++li) {
                const Tile tl = a.tiles[it / a.n_tiles];
                const int j = it % a.n_tiles;
                const int nrows16 = (tl.rows + 15) & ~15;
                // scales / biases of the item's 128 weight rows
                const int sb = li & 1;
                if (!(ok = mbar_wait(&sh.sempty[sb], ((li >> 1) & 1) ^ 1, abort_flag))) break;
                uint8_t* sbuf = scale_base + sb * sbuf_bytes;
                const uint32_t half = (uint32_t)(64 * G * 2);  // bytes of 64 rows
                if (MODE == kGateUp) {
                    const size_t r_gate = (size_t)tl.e * a.N + 64 * j;
                    const size_t r_up = (size_t)tl.e * a.N + a.inter + 64 * j;
                    mbar_arrive_expect_tx(&sh.sfull[sb], 4 * half);
                    bulk_load(sbuf, a.scales + r_gate * G, half, &sh.sfull[sb]);
                    bulk_load(sbuf + half, a.scales + r_up * G, half, &sh.sfull[sb]);
                    bulk_load(sbuf + 2 * half, a.biases + r_gate * G, half, &sh.sfull[sb]);
                    bulk_load(sbuf + 3 * half, a.biases + r_up * G, half, &sh.sfull[sb]);
                } else {
                    const size_t r0 = (size_t)tl.e * a.N + 128 * j;
                    mbar_arrive_expect_tx(&sh.sfull[sb], 4 * half);
                    bulk_load(sbuf, a.scales + r0 * G, 2 * half, &sh.sfull[sb]);
                    bulk_load(sbuf + 2 * half, a.biases + r0 * G, 2 * half, &sh.sfull[sb]);
                }
                for (int s = 0; s < nstages; ++s, ++gs) {
                    const int slot = gs % NS;
                    if (!(ok = mbar_wait(&sh.empty[slot], ((gs / NS) & 1) ^ 1, abort_flag))) break;
                    uint8_t* st = base + (size_t)slot * sbytes;
                    const int kr = min(kStageK, K - s * kStageK);
                    const int atoms = kr / 64;
                    mbar_arrive_expect_tx(&sh.full[slot], kPackedStageBytes + atoms * nrows16 * 128);
                    if (MODE == kGateUp) {
                        tma_load_2d(st, &wmap, &sh.full[slot], s * 32, tl.e * a.N + 64 * j);
                        tma_load_2d(st + 64 * 128, &wmap, &sh.full[slot], s * 32, tl.e * a.N + a.inter + 64 * j);
                    } else {
                        tma_load_2d(st, &wmap, &sh.full[slot], s * 32, tl.e * a.N + 128 * j);
                    }
                    uint8_t* bst = st + kPackedStageBytes;
                    for (int at = 0; at < atoms; ++at)
                        for (int r = 0; r < nrows16; r += 16)
                            tma_load_2d(bst + at * NMAX * 128 + r * 128, &bmap, &sh.full[slot],
                                        s * kStageK + at * 64, tl.p0 + r);
                }
            }
            // Do not leave while copies into shared memory are in flight.
            for (uint32_t g = (gs > (uint32_t)NS ? gs - NS : 0); g < gs; ++g)
                mbar_wait(&sh.full[g % NS], (g / NS) & 1, abort_flag);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer --
        // Each 256-K stage accumulates into a fresh TMEM region (alternating
        // between two); the epilogue adds the stage partials in fp32
        // registers. Short tensor-core accumulation chains keep z close to
        // the exactly rounded value.
        if (lane == 0) {
            uint32_t gs = 0;
            bool ok = true;
            for (int it = blockIdx.x; it < num_items && ok; it += gridDim.x) {
                const Tile tl = a.tiles[it / a.n_tiles];
                const uint32_t nrows16 = (uint32_t)((tl.rows + 15) & ~15);
                const uint32_t idesc = idesc_bf16_m128(nrows16);
                for (int s = 0; s < nstages; ++s, ++gs) {
                    const int slot = gs % NS;
                    const int as = gs & 1;
                    const int pr = gs & 1;
                    if (!(ok = mbar_wait(&sh.full[slot], (gs / NS) & 1, abort_flag))) break;
                    if (!(ok = mbar_wait(&sh.afull[as], (gs >> 1) & 1, abort_flag))) break;
                    if (!(ok = mbar_wait(&sh.pempty[pr], ((gs >> 1) & 1) ^ 1, abort_flag))) break;
                    tc_fence_after();
                    const int kr = min(kStageK, K - s * kStageK);
                    const uint32_t bst = smem_u32(base + (size_t)slot * sbytes + kPackedStageBytes);
                    const uint32_t pcol = tmem + kPCol0 + pr * 128;
                    for (int k16 = 0; k16 < kr / 16; ++k16) {
                        const int at = k16 >> 2, kk = k16 & 3;
                        const uint64_t bdesc = sw128_kmajor_desc(bst + at * NMAX * 128 + kk * 32);
                        umma_ts(pcol, tmem + as * 128 + k16 * 8, bdesc, idesc, k16 > 0 ? 1u : 0u);
                    }
                    umma_commit(&sh.empty[slot]);
                    umma_commit(&sh.aempty[as]);
                    umma_commit(&sh.pfull[pr]);
                }
            }
        }
    } else if (warp >= 4 && warp < 8) {
        // ------------------------------------------------------- dequant --
        const int q = warp & 3;
        int row;  // row in the packed stage and the scale buffer
        if (MODE == kGateUp)
            row = (lane < 16) ? (16 * q + lane) : (64 + 16 * q + (lane - 16));
        else
            row = 32 * q + lane;
        const uint32_t lane_addr = (uint32_t)(32 * q) << 16;
        uint32_t gs = 0;
        int li = 0;
        bool ok = true;
        for (int it = blockIdx.x; it < num_items && ok; it += gridDim.x, ++li) {
            const int sb = li & 1;
            if (!(ok = mbar_wait(&sh.sfull[sb], (li >> 1) & 1, abort_flag))) break;
            const uint16_t* sS = reinterpret_cast<const uint16_t*>(scale_base + sb * sbuf_bytes);
            const uint16_t* sB = sS + 128 * G;
            for (int s = 0; s < nstages; ++s, ++gs) {
                const int slot = gs % NS;
                const int as = gs & 1;
                if (!(ok = mbar_wait(&sh.full[slot], (gs / NS) & 1, abort_flag))) break;
                if (!(ok = mbar_wait(&sh.aempty[as], ((gs >> 1) & 1) ^ 1, abort_flag))) break;
                tc_fence_after();
                const uint8_t* pst = base + (size_t)slot * sbytes + row * 128;
                const int kr = min(kStageK, K - s * kStageK);
                for (int at = 0; at < kr / 64; ++at) {
                    const int g = s * 4 + at;
                    const uint32_t S1 = sS[row * G + g], B1 = sB[row * G + g];
                    const uint32_t S2 = S1 | (S1 << 16), B2 = B1 | (B1 << 16);
                    const uint4 c0 = *reinterpret_cast<const uint4*>(pst + (((2 * at) ^ (row & 7)) << 4));
                    const uint4 c1 = *reinterpret_cast<const uint4*>(pst + (((2 * at + 1) ^ (row & 7)) << 4));
                    const uint32_t wd[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
                    uint32_t r[32];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const uint32_t w = wd[i];
                        const uint32_t sh4[4] = {w, w >> 4, w >> 8, w >> 12};
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const uint32_t t = lop3_and_or(sh4[c], 0x000F000Fu, 0x43004300u);  // 128+q
                            const uint32_t qv = fma_bf16x2(t, 0x3F803F80u, 0xC300C300u);       // q exactly
                            r[4 * i + c] = fma_bf16x2(qv, S2, B2);                            // bf16(S q + B)
                        }
                    }
                    tmem_st32(tmem + lane_addr + as * 128 + at * 32, r);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&sh.afull[as]);
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.empty[slot]);
            }
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(&sh.sempty[sb]);
        }
    } else if (warp >= 8) {
        // ------------------------------------------------------ epilogue --
        const int q = warp & 3;
        const uint32_t lane_addr = (uint32_t)(32 * q) << 16;
        uint32_t gs = 0;
        bool ok = true;
        for (int it = blockIdx.x; it < num_items && ok; it += gridDim.x) {
            const Tile tl = a.tiles[it / a.n_tiles];
            const int j = it % a.n_tiles;
            const int nrows16 = (tl.rows + 15) & ~15;
            float acc[NMAX];
#pragma unroll
            for (int c = 0; c < NMAX; ++c) acc[c] = 0.f;
            for (int s = 0; s < nstages; ++s, ++gs) {
                const int pr = gs & 1;
                if (!(ok = mbar_wait(&sh.pfull[pr], (gs >> 1) & 1, abort_flag))) break;
                tc_fence_after();
#pragma unroll
                for (int c0 = 0; c0 < NMAX; c0 += 16) {
                    if (c0 < nrows16) {
                        uint32_t v[16];
                        tmem_ld16(tmem + lane_addr + kPCol0 + pr * 128 + c0, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) acc[c0 + jj] = __fadd_rn(acc[c0 + jj], __uint_as_float(v[jj]));
                    }
                }
                tc_fence_before();
                mbar_arrive(&sh.pempty[pr]);
            }
            if (!ok) break;
            if (MODE == kGateUp) {
                // lanes 0-15: gate rows, lanes 16-31: up rows of the same n
                const int n = 64 * j + 16 * q + (lane & 15);
                const int pos = interleaved_pos(n);
#pragma unroll
                for (int jj = 0; jj < NMAX; jj += 2) {
                    if (jj < nrows16) {
                        const float send = (lane < 16) ? acc[jj + 1] : acc[jj];
                        const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
                        const int tok = jj + (lane < 16 ? 0 : 1);
                        const float gf = lane < 16 ? acc[jj] : recv;
                        const float uf = lane < 16 ? recv : acc[jj + 1];
                        const float gb = bf16_bits_to_f32(f32_to_bf16_bits(gf));  // z is a bf16 tensor
                        const float ub = bf16_bits_to_f32(f32_to_bf16_bits(uf));
                        if (tok < tl.rows)
                            a.out[(size_t)(tl.p0 + tok) * a.out_ld + pos] = (uint16_t)geglu_bf16(gb, ub);
                    }
                }
            } else {
                const int h = 128 * j + 32 * q + lane;
#pragma unroll
                for (int jj = 0; jj < NMAX; ++jj) {
                    if (jj < tl.rows) {
                        const int f = a.perm[tl.p0 + jj];
                        a.out[(size_t)f * a.out_ld + h] = (uint16_t)f32_to_bf16_bits(acc[jj]);
                    }
                }
            }
        }
    }

    __syncwarp();  // role warps diverge (one elected lane); reconverge before the block barrier
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

size_t gemm_smem_bytes(int mode, int K, int nmax, int stages) {
    (void)mode;
    return 1024 /* alignment slack */ + (size_t)stages * stage_bytes(nmax) + 2 * (size_t)scale_buf_bytes(K);
}

int gemm_max_stages(int mode, int K, int nmax) {
    const size_t limit = 232448 - 2048;  // 227 KB per CTA minus the static part
    int s = 8;
    while (s > 1 && gemm_smem_bytes(mode, K, nmax, s) > limit) --s;
    return s;
}

template <int MODE, int NMAX>
static cudaError_t launch_one(const CUtensorMap& wmap, const CUtensorMap& bmap, const GemmArgs& a, int grid,
                              size_t smem, cudaStream_t stream) {
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        cudaError_t err = cudaFuncSetAttribute(grouped_gemm_kernel<MODE, NMAX>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, 232448 - 2048);
        if (err != cudaSuccess) return err;
        attr_set[dev] = true;
    }
    grouped_gemm_kernel<MODE, NMAX><<<grid, kThreads, smem, stream>>>(wmap, bmap, a);
    return cudaGetLastError();
}

cudaError_t launch_gemm(int mode, const CUtensorMap& wmap, const CUtensorMap& bmap, const GemmArgs& a, int grid,
                        cudaStream_t stream) {
    const size_t smem = gemm_smem_bytes(mode, a.K, a.nmax, a.stages);
    if (a.nmax == 64)
        return mode == kGateUp ? launch_one<kGateUp, 64>(wmap, bmap, a, grid, smem, stream)
                               : launch_one<kDown, 64>(wmap, bmap, a, grid, smem, stream);
    if (a.nmax == 128)
        return mode == kGateUp ? launch_one<kGateUp, 128>(wmap, bmap, a, grid, smem, stream)
                               : launch_one<kDown, 128>(wmap, bmap, a, grid, smem, stream);
    return cudaErrorInvalidValue;
}

int gemm_error_word() {
    int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_error_word, sizeof(int)) != cudaSuccess) return 0;
    cudaMemcpyToSymbol(g_error_word, &z, sizeof(int));
    return v;
}

}  // namespace moe
