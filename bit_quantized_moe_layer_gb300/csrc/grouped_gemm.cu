// Grouped 4-bit dequant-GEMM on the 5th-generation tensor cores (tcgen05):
// the two QuantizedSwitchLinear calls of DiffExperts.forward
// ("diffusion-gemma/model.ts"), gate_up with the split + GeGLU fused into its
// epilogue, and down; with one expert, the dense MLP's linears and the tied
// head (DiffusionGemmaModel.logitsFromHidden), whose epilogue applies the
// final-logit softcap.
//
// The product is computed transposed (D^T = W . X^T) so the weight rows fill
// the 128-row M side of the MMA and the few tokens an expert receives fill
// the N side (16..128): at small token counts every weight byte is read from
// HBM once and the tensor cores stay far from busy.
//
// Persistent kernel, one CTA per SM, work item = (token tile of one expert,
// 128-row weight tile), K in stages of 256. Warp roles:
//   warp 0        TMA producer of the packed weights (128 rows x 128 B per
//                 stage, 128 B swizzle) into a ring of up to 8 stages, and of
//                 the item's scales and biases (bulk copies, double-buffered);
//   warp 1        TMEM owner and MMA issuer (one elected thread): per stage
//                 it waits for the A slot and the B slot, at an item's first
//                 stage for a free accumulator buffer (the 128-row kernel's
//                 token copy completes on the A slot's barrier and one
//                 commit frees both slots: one wait and one commit a stage);
//   warp 2        TMA producer of the B operand into a ring that the MMA's
//                 completion releases: one 3-D copy a stage of its four
//                 64-wide atoms (a box of 16 to 128 rows, the smallest that
//                 holds the tile), the atoms (box rows) x 128 B apart. (The
//                 lockstep kernel for token tiles of up to 64 rows, used
//                 when the weight ring is too shallow for the groups, loads
//                 16-row, 64-wide blocks instead, the atoms brows x 128 B
//                 apart.)
//                 The slots are sized at run time for the largest token
//                 tile of the call, so small tiles get a deep ring;
//   dequant warps thread = weight row = TMEM lane. Token tiles of up to 64
//                 rows: 3 groups of 4 warps (one per TMEM lane quarter);
//                 group r takes every stage g with g % 3 == r, all four
//                 atoms of its quarter, into A slot r, so the two or three
//                 dequant warps sharing a scheduler work on different stages
//                 and one covers the other's barrier waits. Tiles of up to
//                 128 rows: 8 warps in lockstep, warp (q, p) dequantises
//                 atoms 2p and 2p + 1 (64 K each) of lane quarter q of every
//                 stage into the next of 2 A slots. A packed word holds 8
//                 codes; the 0x4300 magic
//                 gives 128+q per bf16 half, minus 128 gives q exactly, and
//                 one fma.rn.bf16x2 with the group's scale and bias gives
//                 bf16(S*q + B) with a single rounding. The MMA reads A from
//                 TMEM and B from shared memory;
//   epilogue      an item accumulates its whole K in one of two TMEM
//     warps       accumulator buffers (fp32); once per item these warps read
//                 it and apply GeGLU (gate_up) or store y by sorted row
//                 (down, through a shared-memory staging tile as 16-byte
//                 pieces of rows) while the next item accumulates in the
//                 other buffer.
// The dequantised pair order inside each 8-element K block is (0,4),(1,5),
// (2,6),(3,7); the B operands (gathered x, GeGLU output) are stored in that
// same K order, so the MMA sums the same products.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kStageK = 256;
constexpr int kPackedStageBytes = 128 * 128;  // 128 rows x 32 words
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxPackedStages = 8;
constexpr int kMaxBStages = 8;
constexpr int kEpiStageBytes = 8 * 1024;  // down epilogue: [16 tokens][32 rows] bf16 per epilogue warp (<= 8)
constexpr int kMaxASlots = 3;  // A-operand ring in TMEM (128 columns a slot)
// Sleep between tests for waits with slack (producers, epilogue).
constexpr uint32_t kSleepRing = 200;  // ns: the TMA producers
constexpr uint32_t kSleepEpi = 1000;  // ns: the epilogue has a whole item of slack

struct Smem {
    uint64_t wfull[kMaxPackedStages], wempty[kMaxPackedStages];  // packed-weight ring
    uint64_t bfull[kMaxBStages], bempty[kMaxBStages];            // B-operand ring
    uint64_t afull[kMaxASlots], aempty[kMaxASlots];              // A slots in TMEM
    uint64_t dfull[2], dempty[2];                                // accumulator buffers in TMEM
    uint64_t sfull[2], sempty[2];                                // scale/bias buffers
    uint64_t mdrain;  // the MMA issuer's final commit
    uint32_t tmem_base;
    int abort_flag;
};

__host__ __device__ inline int scale_buf_bytes(int K) {
    // scales + biases for 128 rows, rounded up to 1 KB
    return ((128 * (K / 64) * 2 * 2) + 1023) & ~1023;
}

// Rows of the B box that holds a tile of `rows` token rows: 16 << index.
__device__ __forceinline__ int bbox_index(int rows) {
    int i = 0;
    while ((16 << i) < rows && i < 3) ++i;
    return i;
}

// Token tile and weight tile of work item `it` (ntok token tiles).
__device__ __forceinline__ void item_coords(const GemmArgs& a, int ntok, int it, int& ti, int& j) {
    if (a.weight_major) {
        ti = it % ntok;
        j = it / ntok;
    } else {
        ti = it / a.n_tiles;
        j = it % a.n_tiles;
    }
}

}  // namespace

// NA A slots in TMEM (a ring the dequant warps fill ahead of the MMA), EPW
// epilogue warps per TMEM lane quarter. GROUPS: NA groups of 4 dequant
// warps, group r taking the stages g with g % NA == r into A slot r (each
// warp all four atoms of its lane quarter); otherwise 16 / APW dequant
// warps in lockstep, APW atoms of every stage each.
template <int NA, int APW, bool GROUPS>
__host__ __device__ constexpr int dequant_warps() {
    return GROUPS ? 4 * NA : 16 / APW;
}

template <int MODE, int NMAX, int NA, int APW, int EPW, bool GROUPS>
__global__ void __launch_bounds__((3 + dequant_warps<NA, APW, GROUPS>() + 4 * EPW) * 32, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ BMaps bmaps,
                        GemmArgs a) {
    constexpr int kDqWarps = dequant_warps<NA, APW, GROUPS>();
    // one 3-D box a token stage (the lockstep kernel for tiles of up to 64
    // rows loads 16-row blocks)
    constexpr bool kBox3 = NMAX > 64 || GROUPS;
    constexpr int kEpiWarp0 = 3 + kDqWarps;
    constexpr int kEpiWarps = 4 * EPW;
    constexpr int kAccChunks = NMAX / 16 / EPW;  // 16-column chunks of one epilogue warp
    constexpr uint32_t kD0 = NA * 128;           // accumulator buffers after the A slots
    static_assert(kD0 + 2 * NMAX <= kTmemCols, "TMEM columns");
    static_assert(NA <= kMaxASlots, "A slots");
    // Merged rings (128-row lockstep kernel): the token operand's ring is
    // the A ring (one slot a stage): its copy completes on the stage's A
    // barrier, and one MMA commit frees both, so the MMA issuer, whose
    // barrier operations delay its MMAs, waits on one barrier and commits
    // once a stage. Taken when NA token slots of the call's size fit in the
    // token region (always: it holds two of the largest). The stage-group
    // kernel keeps its deeper token ring (merged there, with three slots,
    // canvas measured 144.6 -> 146.9 us).
    constexpr bool kMergeable = !GROUPS && NMAX == 128;
    extern __shared__ __align__(1024) uint8_t dsmem[];
    __shared__ Smem sh;
    pdl_trigger();
    // Before waiting for the routing: warm L2 with the weights and scales of
    // this CTA's first items (the preceding kernels leave HBM idle). Only
    // global data that no earlier kernel writes is touched here.
    if (threadIdx.x == 0 && a.prefetch_items > 0) {
        const uint32_t row_bytes = (uint32_t)a.K / 2, G = (uint32_t)a.K / 64;
        for (int i = 0; i < a.prefetch_items; ++i) {
            const int it = blockIdx.x + i * gridDim.x;
            // before the wait the token-tile count is the host's (tiles_per_expert)
            int ti, j;
            item_coords(a, a.tiles_per_expert, it, ti, j);
            const int e = ti / a.tiles_per_expert;
            if (e >= a.E || j >= a.n_tiles) break;  // past the last item
            const int nblk = (MODE == kGateUp) ? 2 : 1;  // gate and up halves, or one 128-row block
            for (int h = 0; h < nblk; ++h) {
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
    // 1024-byte aligned carve-up: packed ring | B ring | 2 scale buffers.
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsmem) + 1023) & ~uintptr_t(1023));
    const int NP = a.wstages;
    // brows: the largest token tile's rows rounded up to a power of two
    // (16..NMAX). It sizes the B slots (4 atoms of brows x 128 B, each atom
    // 1024-byte aligned), so small tiles get a deep B ring.
    const int maxrows = a.num_tiles[1];
    int brows = 16;
    while (brows < maxrows && brows < NMAX) brows <<= 1;
    const int bslot_bytes = 4 * brows * 128;
    const bool merged = kMergeable && NA * bslot_bytes <= a.bregion;  // uniform over the CTA
    const int NB = merged ? NA : min(kMaxBStages, a.bregion / bslot_bytes);
    uint8_t* wring = base;
    uint8_t* bring = base + (size_t)NP * kPackedStageBytes;
    uint8_t* scale_base = bring + (size_t)a.bregion;
    const int G = a.K / 64;  // groups per weight row
    const int sbuf_bytes = scale_buf_bytes(a.K);
    // down: the epilogue's staging tiles after the scale buffers
    uint8_t* epi_stage =
        reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(scale_base + 2 * sbuf_bytes) + 127) & ~uintptr_t(127));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int* abort_flag = &sh.abort_flag;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NP; ++s) {
            mbar_init(&sh.wfull[s], 1);
            mbar_init(&sh.wempty[s], GROUPS ? 4 : kDqWarps);  // the warps that read the stage
        }
        for (int s = 0; s < NB; ++s) {
            mbar_init(&sh.bfull[s], 1);
            mbar_init(&sh.bempty[s], 1);
        }
        for (int i = 0; i < NA; ++i) {
            // the warps that write the slot (and the token copy's arrival)
            mbar_init(&sh.afull[i], (GROUPS ? 4 : kDqWarps) + (merged ? 1 : 0));
            mbar_init(&sh.aempty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sh.sfull[i], 1);
            mbar_init(&sh.sempty[i], kDqWarps);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sh.dfull[i], 1);
            mbar_init(&sh.dempty[i], kEpiWarps);
        }
        mbar_init(&sh.mdrain, 1);
        sh.abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&sh.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;

    const int ntok = a.num_tiles[0];
    const int num_items = ntok * a.n_tiles;
    const int K = a.K;
    const int nstages = (K + kStageK - 1) / kStageK;
    if (warp == 0) {
        // ------------------------------------- packed weights + scales --
        // The whole warp runs the loop; one elected lane issues the copies.
        if (elect_one()) prefetch_tensormap(&wmap);
        int slot = 0;
        uint32_t ph = 0, issued = 0;
        int li = 0;
        bool ok = true;
        for (int it = blockIdx.x; it < num_items && ok; it += gridDim.x, ++li) {
            int ti, j;
            item_coords(a, ntok, it, ti, j);
            const Tile tl = a.tiles[ti];
            const int sb = li & 1;
            if (!(ok = mbar_wait(&sh.sempty[sb], ((li >> 1) & 1) ^ 1, abort_flag, kSleepRing, 1))) break;
            uint8_t* sbuf = scale_base + sb * sbuf_bytes;
            const uint32_t half = (uint32_t)(64 * G * 2);  // bytes of 64 rows
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
        for (int l = (li > 2 ? li - 2 : 0); l < li; ++l) mbar_drain(&sh.sfull[l & 1], (l >> 1) & 1);
    } else if (warp == 2) {
        // ---------------------------------------------------- B operand --
        if (elect_one()) {
            for (int i = 0; i < 4; ++i) prefetch_tensormap(&bmaps.m[i]);
            prefetch_tensormap(&bmaps.m2);
        }
        const uint32_t box_atoms = (uint32_t)min(4, K / 64);
        uint64_t* const bF = merged ? sh.afull : sh.bfull;    // the copy completes here
        uint64_t* const bE = merged ? sh.aempty : sh.bempty;  // the slot is free
        int slot = 0;
        uint32_t ph = 0, issued = 0;
        bool ok = true;
        for (int it = blockIdx.x; it < num_items && ok; it += gridDim.x) {
            int ti, j;
            item_coords(a, ntok, it, ti, j);
            const Tile tl = a.tiles[ti];
            const int bi = bbox_index(tl.rows);
            const int nrows16 = (tl.rows + 15) & ~15;
            // the whole box counts, rows and atoms past the tensor (zero-filled) included
            const uint32_t box_bytes = box_atoms * (16u << bi) * 128u;
            for (int s = 0; s < nstages; ++s) {
                if (!(ok = mbar_wait(&bE[slot], ph ^ 1, abort_flag, kSleepRing, 3))) break;
                uint8_t* bst = bring + (size_t)slot * bslot_bytes;
                if (elect_one()) {
                    if constexpr (kBox3) {
                        mbar_arrive_expect_tx(&bF[slot], box_bytes);
                        tma_load_3d(bst, &bmaps.m[bi], &bF[slot], 0, tl.p0, s * (kStageK / 64));
                    } else {
                        const int atoms = min(kStageK, K - s * kStageK) / 64;
                        mbar_arrive_expect_tx(&bF[slot], atoms * nrows16 * 128);
                        for (int at = 0; at < atoms; ++at)
                            for (int r = 0; r < nrows16; r += 16)
                                tma_load_2d(bst + at * brows * 128 + r * 128, &bmaps.m2, &bF[slot],
                                            s * kStageK + at * 64, tl.p0 + r);
                    }
                }
                __syncwarp();
                ++issued;
                if (++slot == NB) {
                    slot = 0;
                    ph ^= 1;
                }
            }
        }
        for (uint32_t g = (issued > (uint32_t)NB ? issued - NB : 0); g < issued; ++g)
            mbar_drain(&bF[g % NB], (g / NB) & 1);
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer --
        // The whole warp runs the loop; one elected lane issues the MMAs of a
        // stage and the commits (a commit tracks its own thread's MMAs). An
        // item accumulates its whole K into accumulator buffer li & 1.
        int bslot = 0, li = 0, as = 0;
        uint32_t bph = 0, aph = 0;  // phases of the B slot's and the A slot's barriers
        bool ok = true;
        // Token rows of this CTA's items li and li + 32 in lane li % 32,
        // loaded once: the issuer paces the whole pipeline, and a global load
        // at each item boundary cost it ~500 cycles an item (measured with a
        // per-stage clock trace). Items from the 64th on (long weight-major
        // calls) load their rows one item ahead instead.
        int rows_lo = 0, rows_hi = 0, rows_next = 0;
        {
            int ti, jn;
            const int i0 = blockIdx.x + lane * (int)gridDim.x, i1 = i0 + 32 * (int)gridDim.x;
            if (i0 < num_items) {
                item_coords(a, ntok, i0, ti, jn);
                rows_lo = a.tiles[ti].rows;
            }
            if (i1 < num_items) {
                item_coords(a, ntok, i1, ti, jn);
                rows_hi = a.tiles[ti].rows;
            }
        }
        for (int it = blockIdx.x; it < num_items && ok; it += gridDim.x, ++li) {
            const int r_lo = __shfl_sync(0xffffffffu, rows_lo, li & 31);
            const int r_hi = __shfl_sync(0xffffffffu, rows_hi, li & 31);
            const int rows = li < 32 ? r_lo : (li < 64 ? r_hi : rows_next);
            if (li >= 63 && it + (int)gridDim.x < num_items) {
                int ti, jn;
                item_coords(a, ntok, it + gridDim.x, ti, jn);
                rows_next = a.tiles[ti].rows;
            }
            const uint32_t nrows16 = (uint32_t)((rows + 15) & ~15);
            const uint32_t idesc = idesc_bf16_m128(nrows16);
            // distance of the B slot's atoms in descriptor units (16 B)
            const uint32_t atom_step =
                (uint32_t)((kBox3 ? (16 << bbox_index(rows)) : brows) * 128) >> 4;
            const int db = li & 1;
            const uint32_t dcol = tmem + kD0 + (uint32_t)(db * NMAX);
            // the accumulator buffer's previous item (li - 2) has been read out
            if (li >= 2 && !(ok = mbar_wait(&sh.dempty[db], ((li >> 1) - 1) & 1, abort_flag, 0, 6))) break;
            for (int s = 0; s < nstages; ++s) {
                if (!(ok = mbar_wait(&sh.afull[as], aph, abort_flag, 0, 7))) break;
                if (!merged && !(ok = mbar_wait(&sh.bfull[bslot], bph, abort_flag, 0, 5))) break;
                tc_fence_after();
                const int nk = min(kStageK, K - s * kStageK) / 16;
                const uint64_t bdesc0 = sw128_kmajor_desc(smem_u32(bring + (size_t)bslot * bslot_bytes));
                const uint32_t acol = tmem + as * 128;
                if (elect_one()) {
                    if (nk == 16) {
                        // a full stage: 16 MMAs without a per-MMA test (the
                        // tests slowed the issuer, which paces the pipeline)
                        const uint64_t b1 = bdesc0 + atom_step, b2 = b1 + atom_step, b3 = b2 + atom_step;
                        umma_ts(dcol, acol + 0, bdesc0 + 0, idesc, s > 0 ? 1u : 0u);
                        umma_ts(dcol, acol + 8, bdesc0 + 2, idesc, 1u);
                        umma_ts(dcol, acol + 16, bdesc0 + 4, idesc, 1u);
                        umma_ts(dcol, acol + 24, bdesc0 + 6, idesc, 1u);
                        umma_ts(dcol, acol + 32, b1 + 0, idesc, 1u);
                        umma_ts(dcol, acol + 40, b1 + 2, idesc, 1u);
                        umma_ts(dcol, acol + 48, b1 + 4, idesc, 1u);
                        umma_ts(dcol, acol + 56, b1 + 6, idesc, 1u);
                        umma_ts(dcol, acol + 64, b2 + 0, idesc, 1u);
                        umma_ts(dcol, acol + 72, b2 + 2, idesc, 1u);
                        umma_ts(dcol, acol + 80, b2 + 4, idesc, 1u);
                        umma_ts(dcol, acol + 88, b2 + 6, idesc, 1u);
                        umma_ts(dcol, acol + 96, b3 + 0, idesc, 1u);
                        umma_ts(dcol, acol + 104, b3 + 2, idesc, 1u);
                        umma_ts(dcol, acol + 112, b3 + 4, idesc, 1u);
                        umma_ts(dcol, acol + 120, b3 + 6, idesc, 1u);
                    } else {
#pragma unroll
                        for (int k16 = 0; k16 < 16; ++k16) {
                            if (k16 < nk) {
                                const uint64_t bdesc = bdesc0 + (uint64_t)((k16 >> 2) * atom_step + (k16 & 3) * 2);
                                umma_ts(dcol, acol + k16 * 8, bdesc, idesc, (s > 0 || k16 > 0) ? 1u : 0u);
                            }
                        }
                    }
                    if (!merged) umma_commit(&sh.bempty[bslot]);
                    umma_commit(&sh.aempty[as]);
                    if (s == nstages - 1) umma_commit(&sh.dfull[db]);
                }
                __syncwarp();
                if (++bslot == NB) {
                    bslot = 0;
                    bph ^= 1;
                }
                if (++as == NA) {
                    as = 0;
                    aph ^= 1;
                }
            }
        }
        // Every MMA this thread issued completes before TMEM is released.
        if (elect_one()) umma_commit(&sh.mdrain);
        __syncwarp();
        mbar_drain(&sh.mdrain, 0);
    } else if (GROUPS && warp >= 3 && warp < kEpiWarp0) {
        // ------------------------------------------- dequant, stage groups --
        // Warp (q, r): TMEM lanes 32q..32q+31 (q = warp % 4, the lane quarter
        // a warp may access), every stage g (counted over this CTA's items)
        // with g % NA == r, all four atoms, into A slot r. Phase safety: a
        // group waits for stage g's weights only after the MMA of stage
        // g - 2 NA has completed (its previous stage waited for that A slot),
        // so every stage up to g - 2 NA has landed; the host launches this
        // kernel only with at least 2 NA weight stages, so the slot of stage
        // g is at most one phase behind when the group waits on it.
        const int q = warp & 3;
        const int grp = (warp - 3) >> 2;
        int row;  // row in the packed stage and the scale buffer
        if (MODE == kGateUp)
            row = (lane < 16) ? (16 * q + lane) : (64 + 16 * q + (lane - 16));
        else
            row = 32 * q + lane;
        const uint32_t lane_addr = (uint32_t)(32 * q) << 16;
        // this thread's 128-byte row in ring slot 0, its 8 chunks swizzled
        uint32_t wo[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            wo[i] = smem_u32(wring) + (uint32_t)row * 128u + ((uint32_t)(i ^ (row & 7)) << 4);
        const uint32_t srow = smem_u32(scale_base) + (uint32_t)(row * G) * 2u;
        const uint32_t bias_off = (uint32_t)(128 * G * 2);
        const uint32_t acol = tmem + lane_addr + (uint32_t)grp * 128u;
        bool ok = true;
        int li = 0;
        uint32_t gbase = 0;  // stages of this CTA's earlier items
        for (int it = blockIdx.x; it < num_items && ok; it += gridDim.x, ++li, gbase += (uint32_t)nstages) {
            const int sb = li & 1;
            if (!(ok = mbar_wait(&sh.sfull[sb], (li >> 1) & 1, abort_flag, 0, 8))) break;
            const uint32_t sS = srow + (uint32_t)(sb * sbuf_bytes);
            const int s0 = (grp - (int)(gbase % NA) + NA) % NA;  // first stage of the item that is ours
            if (s0 >= nstages) mbar_arrive_lane0(&sh.sempty[sb]);  // none: release the scales at once
            for (int s = s0; s < nstages; s += NA) {
                const uint32_t g = gbase + (uint32_t)s;
                const int atoms = min(kStageK, K - s * kStageK) / 64;
                const uint32_t wslot = g % (uint32_t)NP;
                if (!(ok = mbar_wait(&sh.wfull[wslot], (g / NP) & 1, abort_flag, 0, 9))) break;
                uint4 c[8];
                uint32_t S1[4], B1[4];
                const uint32_t so = wslot * (uint32_t)kPackedStageBytes;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if (i < atoms) {  // warp-uniform
                        c[2 * i] = lds128(wo[2 * i] + so);
                        c[2 * i + 1] = lds128(wo[2 * i + 1] + so);
                        S1[i] = lds_u16(sS + (uint32_t)(8 * s + 2 * i));
                        B1[i] = lds_u16(sS + bias_off + (uint32_t)(8 * s + 2 * i));
                    }
                }
                // The arrive releases the loads above: the slot (and, after
                // this warp's last stage of the item, the scale buffer) may
                // be refilled.
                __syncwarp();
                mbar_arrive_lane0(&sh.wempty[wslot]);
                if (s + NA >= nstages) mbar_arrive_lane0(&sh.sempty[sb]);
                if (!(ok = mbar_wait(&sh.aempty[grp], ((g / NA) & 1) ^ 1, abort_flag, 0, 10))) break;
                tc_fence_after();
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if (i < atoms) {
                        uint32_t r[32];
                        dequant_atom(c[2 * i], c[2 * i + 1], S1[i], B1[i], r);
                        tmem_st32(acol + i * 32, r);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                mbar_arrive_lane0(&sh.afull[grp]);
            }
        }
        tmem_wait_st();
    } else if (!GROUPS && warp >= 3 && warp < kEpiWarp0) {
        // ------------------------------------------------------- dequant --
        // 16 / APW warps; warp (q, p) covers TMEM lanes 32q..32q+31 (q =
        // warp % 4, the lane quarter a warp may access) and atoms p APW ..
        // p APW + APW - 1 (64 K each) of every stage. Each stage goes into the
        // next A slot of the ring, so the warps run up to NA stages ahead of
        // the MMA.
        const int dw = warp - 3;
        const int q = warp & 3;
        const int at0 = (dw >> 2) * APW;
        int row;  // row in the packed stage and the scale buffer
        if (MODE == kGateUp)
            row = (lane < 16) ? (16 * q + lane) : (64 + 16 * q + (lane - 16));
        else
            row = 32 * q + lane;
        const uint32_t lane_addr = (uint32_t)(32 * q) << 16;
        // shared addresses: this thread's 128-byte row in ring slot 0 with
        // the swizzled offsets of its atoms, and its scale in buffer 0
        uint32_t wo[2 * APW];
#pragma unroll
        for (int i = 0; i < APW; ++i) {
            const int at = at0 + i;
            wo[2 * i] = smem_u32(wring) + (uint32_t)row * 128u + ((uint32_t)((2 * at) ^ (row & 7)) << 4);
            wo[2 * i + 1] = smem_u32(wring) + (uint32_t)row * 128u + ((uint32_t)((2 * at + 1) ^ (row & 7)) << 4);
        }
        const uint32_t srow = smem_u32(scale_base) + (uint32_t)(row * G + at0) * 2u;
        const uint32_t bias_off = (uint32_t)(128 * G * 2);
        int wslot = 0, as = 0;
        uint32_t wph = 0, aph = 0;
        bool ok = true;
        int li = 0;
        for (int it = blockIdx.x; it < num_items && ok; it += gridDim.x, ++li) {
            const int sb = li & 1;
            if (!(ok = mbar_wait(&sh.sfull[sb], (li >> 1) & 1, abort_flag, 0, 8))) break;
            const uint32_t sS = srow + (uint32_t)(sb * sbuf_bytes);
            for (int s = 0; s < nstages; ++s) {
                const int atoms = min(kStageK, K - s * kStageK) / 64;
                if (!(ok = mbar_wait(&sh.wfull[wslot], wph, abort_flag, 0, 9))) break;
                uint4 c[2 * APW];
                uint32_t S1[APW], B1[APW];
                const uint32_t so = (uint32_t)(wslot * kPackedStageBytes);
#pragma unroll
                for (int i = 0; i < APW; ++i) {
                    if (at0 + i < atoms) {  // warp-uniform
                        c[2 * i] = lds128(wo[2 * i] + so);
                        c[2 * i + 1] = lds128(wo[2 * i + 1] + so);
                        S1[i] = lds_u16(sS + (uint32_t)(8 * s + 2 * i));
                        B1[i] = lds_u16(sS + bias_off + (uint32_t)(8 * s + 2 * i));
                    }
                }
                // The arrive releases the loads above: the slot (and, after
                // the item's last stage, the scale buffer) may be refilled.
                __syncwarp();
                mbar_arrive_lane0(&sh.wempty[wslot]);
                if (s == nstages - 1) mbar_arrive_lane0(&sh.sempty[sb]);
                if (++wslot == NP) {
                    wslot = 0;
                    wph ^= 1;
                }
                if (!(ok = mbar_wait(&sh.aempty[as], aph ^ 1, abort_flag, 0, 10))) break;
                tc_fence_after();
#pragma unroll
                for (int i = 0; i < APW; ++i) {
                    if (at0 + i < atoms) {
                        uint32_t r[32];
                        dequant_atom(c[2 * i], c[2 * i + 1], S1[i], B1[i], r);
                        tmem_st32(tmem + lane_addr + as * 128 + (at0 + i) * 32, r);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                mbar_arrive_lane0(&sh.afull[as]);
                if (++as == NA) {
                    as = 0;
                    aph ^= 1;
                }
            }
        }
        tmem_wait_st();
    } else if (warp >= kEpiWarp0) {
        // ------------------------------------------------------ epilogue --
        // Warp (q, h): TMEM lanes 32q..32q+31, the 16-column chunks h, h+EPW, ...
        const int q = warp & 3;
        const int h = (warp - kEpiWarp0) >> 2;
        const uint32_t lane_addr = (uint32_t)(32 * q) << 16;
        bool ok = true;
        int li = 0;
        for (int it = blockIdx.x; it < num_items && ok; it += gridDim.x, ++li) {
            int ti, j;
            item_coords(a, ntok, it, ti, j);
            const Tile tl = a.tiles[ti];
            const int nrows16 = (tl.rows + 15) & ~15;
            // The item's accumulator (buffer li & 1) holds the whole K: this
            // warp reads its 16-column chunks one at a time, then hands the
            // buffer back (it is not needed again before item li + 2).
            const int db = li & 1;
            if (!(ok = mbar_wait(&sh.dfull[db], (li >> 1) & 1, abort_flag, kSleepEpi, 11))) break;
            tc_fence_after();
            const uint32_t dcol = tmem + lane_addr + kD0 + (uint32_t)(db * NMAX);
            // Not unrolled: the epilogue has a whole item of slack, and its
            // unrolled body (GeGLU or the softcap for every chunk) crowded the
            // dequantisation and MMA loops out of the instruction cache
            // (measured: canvas step 183 -> 176 us, prefill 731 -> 637 us).
#pragma unroll 1
            for (int cl = 0; cl < kAccChunks; ++cl) {
                const int c0 = (cl * EPW + h) * 16;
                if (c0 >= nrows16) continue;  // warp-uniform
                uint32_t raw[16];
                tmem_ld16(dcol + c0, raw);
                tmem_wait_ld();
                float v[16];
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) v[jj] = __uint_as_float(raw[jj]);
                if (MODE == kGateUp) {
                    // lanes 0-15: gate rows, lanes 16-31: up rows of the same n
                    const int pos = interleaved_pos(64 * j + 16 * q + (lane & 15));
#pragma unroll
                    for (int jj = 0; jj < 16; jj += 2) {
                        const float send = (lane < 16) ? v[jj + 1] : v[jj];
                        const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
                        const int tok = c0 + jj + (lane < 16 ? 0 : 1);
                        const float gf = lane < 16 ? v[jj] : recv;
                        const float uf = lane < 16 ? recv : v[jj + 1];
                        const float gb = bf16_bits_to_f32(f32_to_bf16_bits(gf));  // z is a bf16 tensor
                        const float ub = bf16_bits_to_f32(f32_to_bf16_bits(uf));
                        if (tok < tl.rows)
                            a.out[(size_t)(tl.p0 + tok) * a.out_ld + pos] = (uint16_t)geglu_bf16(gb, ub);
                    }
                } else if (MODE == kHead) {
                    // logits bf16 (the head's output dtype), widened to fp32, then
                    // cap * tanh(x / cap) in fp32 steps; 32 lanes store 128 B of a row
                    const int vrow = 128 * j + 32 * q + lane;
                    const float cap = a.softcap;
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int tok = c0 + jj;
                        const float x = bf16_bits_to_f32(f32_to_bf16_bits(v[jj]));
                        const float o = cap > 0.f ? __fmul_rn(tanhf(__fdiv_rn(x, cap)), cap) : x;
                        if (tok < tl.rows) a.out_f32[(size_t)(tl.p0 + tok) * a.out_ld + vrow] = o;
                    }
                } else {
                    // y by sorted row, through this warp's [16 tokens][32 rows]
                    // staging tile: the lanes write their row's 16 tokens, then
                    // each lane stores 8 consecutive rows of one token (16
                    // bytes). With one 2-byte store a lane per token the
                    // stores paced the down kernel at T = 4096 (149.5 -> 129.0
                    // us measured; canvas 47.1 -> 45.1).
                    uint16_t* stg = reinterpret_cast<uint16_t*>(epi_stage + (size_t)(warp - kEpiWarp0) * 1024);
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) stg[jj * 32 + lane] = (uint16_t)f32_to_bf16_bits(v[jj]);
                    __syncwarp();
                    const int hbase = 128 * j + 32 * q;
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int tokl = (lane >> 2) + 8 * u, seg = lane & 3;
                        const uint4 val = *reinterpret_cast<const uint4*>(stg + tokl * 32 + seg * 8);
                        const int tok = c0 + tokl;
                        if (tok < tl.rows)
                            *reinterpret_cast<uint4*>(a.out + (size_t)(tl.p0 + tok) * a.out_ld + hbase + seg * 8) = val;
                    }
                    __syncwarp();
                }
            }
            tc_fence_before();
            __syncwarp();
            mbar_arrive_lane0(&sh.dempty[db]);
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

size_t gemm_smem_bytes(int mode, int K, int wstages, int bregion) {
    return 1024 /* alignment slack */ + (size_t)wstages * kPackedStageBytes + (size_t)bregion +
           2 * (size_t)scale_buf_bytes(K) + (mode == kDown ? kEpiStageBytes + 128 : 0);
}

// Shared-memory split: the deepest packed-weight ring (up to 8 stages) that
// leaves the B ring at least two slots of the largest possible token tile;
// the rest goes to the B ring.
void gemm_stages(int mode, int K, int nmax, int* wstages, int* bregion) {
    const size_t limit = 232448 - 2048;  // 227 KB per CTA minus the static part
    const int min_b = 2 * 4 * nmax * 128;
    int nw = kMaxPackedStages;
    while (nw > 2 && gemm_smem_bytes(mode, K, nw, min_b) > limit) --nw;
    *wstages = nw;
    *bregion = (int)((limit - gemm_smem_bytes(mode, K, nw, 0)) & ~size_t(1023));
}

template <int MODE, int NMAX, int NA, int APW, int EPW, bool GROUPS>
static cudaError_t launch_one(const CUtensorMap& wmap, const BMaps& bmaps, const GemmArgs& a, int grid,
                              size_t smem, cudaStream_t stream) {
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    auto kernel = grouped_gemm_kernel<MODE, NMAX, NA, APW, EPW, GROUPS>;
    if (!attr_set[dev]) {
        cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448 - 2048);
        if (err != cudaSuccess) return err;
        attr_set[dev] = true;
    }
    constexpr int warps = 3 + dequant_warps<NA, APW, GROUPS>() + 4 * EPW;
    return launch_pdl(kernel, dim3(grid), dim3(warps * 32), smem, stream, wmap, bmaps, a);
}

template <int MODE>
static cudaError_t launch_mode(const CUtensorMap& wmap, const BMaps& bmaps, const GemmArgs& a, int grid,
                               size_t smem, cudaStream_t stream) {
    // Token tiles of up to 128 rows: two A slots (TMEM holds 2 x 128
    // accumulator columns), eight lockstep dequant warps of two atoms each
    // and 8 epilogue warps, as a 128-token tile's GeGLU needs the wider
    // epilogue (19 warps; stage groups measured no faster here).
    //
    // Token tiles of up to 64 rows: three stage groups of four dequant warps
    // (12), one 3-D token box a stage (canvas gate_up 90 -> 76 us, down 51
    // -> 47, decode gate_up 43 -> 37, measured standalone), when the weight
    // ring holds at least 6 stages (the groups' phase-safety condition);
    // otherwise the lockstep kernel.
    if (a.nmax == 64) {
        if (a.wstages >= 2 * 3) return launch_one<MODE, 64, 3, 2, 1, true>(wmap, bmaps, a, grid, smem, stream);
        return launch_one<MODE, 64, 3, 2, 1, false>(wmap, bmaps, a, grid, smem, stream);
    }
    if (a.nmax == 128) return launch_one<MODE, 128, 2, 2, 2, false>(wmap, bmaps, a, grid, smem, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_gemm(int mode, const CUtensorMap& wmap, const BMaps& bmaps, const GemmArgs& a, int grid,
                        cudaStream_t stream) {
    const size_t smem = gemm_smem_bytes(mode, a.K, a.wstages, a.bregion);
    switch (mode) {
        case kGateUp: return launch_mode<kGateUp>(wmap, bmaps, a, grid, smem, stream);
        case kDown: return launch_mode<kDown>(wmap, bmaps, a, grid, smem, stream);
        case kHead: return launch_mode<kHead>(wmap, bmaps, a, grid, smem, stream);
        default: return cudaErrorInvalidValue;
    }
}

int gemm_error_word() {
    int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_error_word, sizeof(int)) != cudaSuccess) return 0;
    cudaMemcpyToSymbol(g_error_word, &z, sizeof(int));
    return v;
}

}  // namespace moe
