// Device helpers shared by the libmoe kernels: bf16 rounding, mbarriers,
// TMA (cp.async.bulk), tcgen05 (TMEM alloc / ld / st / mma / commit), and
// the bounded wait that every pipeline spin goes through.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// ------------------------------------------------------------------ errors --
// Device error word, one per translation unit (and device): bit 0 a
// pipeline wait timed out, bit 1 an expert id was out of range. Each unit
// exports a host function that reads and clears its copy; moe_device_error()
// ORs them together.
static __device__ int g_error_word;

constexpr int kErrTimeout = 1;
constexpr int kErrBadExpert = 2;
// Bits 8..15 of the error word: which wait timed out first (0: none).
constexpr int kErrWhereShift = 8;

// ------------------------------------------------------------------- bf16 --
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

// fp32 -> bf16 bits, round to nearest even (inputs here are finite).
__device__ __forceinline__ uint32_t f32_to_bf16_bits(float f) {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// Two fp32 -> packed bf16x2 (lo in bits 0..15), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Packed bf16 product, each half exact in fp32 and rounded once to nearest even.
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// ---------------------------------------------------------------- smem ptr --
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// --------------------------------------------------------------- mbarrier --
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Arrive from lane 0 of the warp only (a predicated instruction, no branch).
// Call after __syncwarp() so the other lanes' accesses are ordered before it.
__device__ __forceinline__ void mbar_arrive_lane0(uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b32 l;\n\t"
        "mov.u32 l, %%laneid;\n\t"
        "setp.eq.u32 p, l, 0;\n\t"
        "@p mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];\n\t}" ::"r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t saddr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(saddr)
                 : "memory");
    return v;
}

__device__ __forceinline__ uint32_t lds_u16(uint32_t saddr) {
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(saddr) : "memory");
    return v;
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// try_wait with a suspend-time hint: the warp sleeps in hardware until the
// phase completes or about `ns` nanoseconds pass, issuing nothing meanwhile.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}

// Bounded wait on an mbarrier phase. After one plain test the warp sleeps
// between tests, so a waiting warp takes (almost) no issue slots from the
// warps that work: with sleep_ns == 0 in hardware (try_wait with a suspend
// hint: woken soon after the phase completes, for waits on the critical
// path), otherwise for sleep_ns between tests (for warps with slack).
// Returns false if the phase has not completed within ~2 s (then it raises
// the device error word and the CTA's shared abort flag) or if another warp
// of the CTA has already aborted, so a broken pipeline ends the kernel
// instead of hanging the GPU. Callers treat false as "stop issuing work and
// fall through to the exit path".
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          uint32_t sleep_ns = 0, int where = 0) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t n = 1;; ++n) {
        if (sleep_ns == 0) {
            if (mbar_try_wait_sleep(bar, parity, 100000u)) return true;
        } else {
            __nanosleep(sleep_ns);
            if (mbar_try_wait(bar, parity)) return true;
        }
        if ((n & 15u) == 0) {  // the abort flag and the clock, every 16th test
            if (*abort_flag) return false;
            if (global_timer_ns() - t0 > 2000000000ull) {
                *abort_flag = 1;
                atomicOr(&g_error_word, kErrTimeout);
                atomicCAS(&g_error_word, kErrTimeout, kErrTimeout | ((where & 0xFF) << kErrWhereShift));
                return false;
            }
        }
    }
}

// Exit-path wait for this CTA's own asynchronous work (TMA copies into its
// shared memory, MMAs into its TMEM) to finish before the CTA releases that
// memory or exits. It ignores the abort flag (the work completes on its own
// once issued) and gives up after ~200 ms.
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return;
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        __nanosleep(1000);
        if (global_timer_ns() - t0 > 200000000ull) {
            atomicOr(&g_error_word, kErrTimeout);
            return;
        }
    }
}

// ------------------------------------------------------------------- TMA --
// 2-D tiled load of a box into shared memory, completing on `bar`.
// c0 is the innermost coordinate (elements), c1 the row.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0,
                                            int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                                            int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// Untiled bulk copy global -> shared (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Fetch [src, src + bytes) into L2 (bytes a multiple of 16); no completion.
__device__ __forceinline__ void prefetch_l2_bulk(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// --------------------------------------------------------------- tcgen05 --
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16 (bf16 in, fp32 accumulate).
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (bf16 in, fp32 accumulate).
__device__ __forceinline__ void umma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on `bar` once all tcgen05 async ops issued so far by this thread complete.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Each thread of the warp writes 32 consecutive 32-bit columns of its lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
        "%13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, "
        "%32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
        "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
        "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

// Each thread of the warp reads 16 consecutive 32-bit columns of its lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
        "%13, %14, %15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]),
          "=r"(v[15])
        : "r"(taddr)
        : "memory");
}

// Shared-memory matrix descriptor for a K-major operand in the 128-byte
// swizzled layout: rows of 128 B (64 bf16 of K), 8-row groups 1024 B apart,
// 16-byte chunks of row r permuted by XOR with (r & 7). The tile base must
// be 1024-byte aligned; stepping K by 16 elements inside the 128-byte row
// adds 32 bytes to the start address.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);          // start address
    d |= (uint64_t)1 << 16;                          // leading byte offset (unused here)
    d |= (uint64_t)(1024 >> 4) << 32;                // stride byte offset: 8 rows * 128 B
    d |= (uint64_t)1 << 46;                          // descriptor version (sm_100 family)
    d |= (uint64_t)2 << 61;                          // swizzle: 128 B
    return d;
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major,
// M = 128, N = n (multiple of 16, <= 256).
__device__ __forceinline__ uint32_t idesc_bf16_m128(uint32_t n) {
    return (1u << 4)              // D format fp32
           | (1u << 7)            // A format bf16
           | (1u << 10)           // B format bf16
           | ((n >> 3) << 17)     // N / 8
           | ((128u >> 4) << 24); // M / 16
}

// ------------------------------------------------------------ misc ------
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));  // (a & b) | c
    return d;
}

__device__ __forceinline__ uint32_t fma_bf16x2(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// One lane of a converged warp (elect.sync). Issue TMA and tcgen05 work from
// inside `if (elect_one())` in a loop the whole warp runs: the operands stay
// warp-uniform, which keeps the issue cost of each instruction low.
__device__ __forceinline__ uint32_t elect_one() {
    uint32_t pred = 0;
    asm volatile(
        "{\n\t.reg .b32 rx;\n\t.reg .pred px;\n\telect.sync rx|px, 0xffffffff;\n\tselp.b32 %0, 1, 0, px;\n\t}"
        : "=r"(pred));
    return pred;
}

// Programmatic dependent launch: let the next kernel of the stream be
// scheduled now (it still waits for this grid before touching memory), and
// wait for the previous kernel's grid to complete and its memory to be
// visible. Both are no-ops for a launch without the programmatic attribute.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Cluster-wide barrier (all threads of all CTAs of the cluster). Non-aligned
// form; callers still reconverge their warp first (__syncwarp).
__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// ------------------------------------------------------ GeGLU, K order --
// bf16(gelu_approx(g) * up) for bf16 g, up, where gelu_approx(g) =
// 0.5 g (1 + tanh(s)), s = sqrt(2/pi) (g + 0.044715 g^3). 0.5 (1 + tanh s) is
// the logistic of 2s, evaluated in that form so it keeps its relative
// accuracy where 1 + tanh(s) cancels (s << 0). p = g*up is exact in fp32.
// r = e / (1 + e) with e = exp(-2|s|): for s < 0 it is the logistic of 2s
// and the value is p r; for s >= 0 it is 1 - logistic(2s) > 0 and the value
// is p - p r, formed by a fused multiply-add rounded toward zero: the exact
// value lies strictly between 0 and p, so an exact bf16 tie of p (large g,
// where r is below fp32's resolution of 1) rounds toward zero as the exact
// value does. One exp and one divide serve both signs. For e <= 2^-25,
// 1 + e rounds to 1 and the quotient is e itself: taking e skips the
// divide's slow path for subnormal e (far tails of s), with the same result.
__device__ __forceinline__ uint32_t geglu_bf16(float g, float up) {
    const float c = 0.7978845608028654f;  // sqrt(2/pi)
    const float s = __fmul_rn(c, __fadd_rn(g, __fmul_rn(0.044715f, __fmul_rn(g, __fmul_rn(g, g)))));
    const float p = __fmul_rn(g, up);
    const float e = expf(__fmul_rn(-2.0f, fabsf(s)));
    const float r = (e <= 0x1p-25f) ? e : __fdiv_rn(e, __fadd_rn(1.0f, e));
    const float m = (s < 0.f) ? __fmul_rn(p, r) : __fmaf_rz(-p, fmaxf(r, 1e-30f), p);
    return f32_to_bf16_bits(m);
}

// Position of element n inside its 8-block in the interleaved K order.
__device__ __forceinline__ int interleaved_pos(int n) {
    const int r = n & 7;
    return (n & ~7) | (r < 4 ? 2 * r : 2 * r - 7);
}

// ------------------------------------------------------------- dequant --
// Dequantise one 64-wide K atom (8 packed words) of a weight row with its
// group's scale and bias (bf16 bits) into 32 bf16x2 TMEM columns.
__device__ __forceinline__ void dequant_atom(const uint4 c0, const uint4 c1, uint32_t S1, uint32_t B1,
                                             uint32_t (&r)[32]) {
    const uint32_t S2 = S1 | (S1 << 16), B2 = B1 | (B1 << 16);
    const uint32_t wd[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
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
}

// ------------------------------------------------------------ row norms --
// 8 bf16 (one 16-byte chunk) -> positions holding elements (0,4,1,5,2,6,3,7):
// the K order in which the grouped GEMM's dequantised weights come out.
__device__ __forceinline__ uint4 interleave8(uint4 v) {
    uint4 o;
    o.x = __byte_perm(v.x, v.z, 0x5410);
    o.y = __byte_perm(v.x, v.z, 0x7632);
    o.z = __byte_perm(v.y, v.w, 0x5410);
    o.w = __byte_perm(v.y, v.w, 0x7632);
    return o;
}

// Error-free sum a + b = s + e (Knuth's two-sum).
__device__ __forceinline__ void two_sum_f(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    const float bp = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp));
}

// Adds the squares of both bf16 halves of `b` (exact in fp32) to the
// two-float sum (hi, lo).
__device__ __forceinline__ void sumsq_bf16x2(uint32_t b, float& hi, float& lo) {
    const float l = __uint_as_float(b << 16), h = __uint_as_float(b & 0xFFFF0000u);
    float s1, e1;
    two_sum_f(hi, __fmul_rn(l, l), s1, e1);
    hi = s1;
    lo = __fadd_rn(lo, e1);
    two_sum_f(hi, __fmul_rn(h, h), s1, e1);
    hi = s1;
    lo = __fadd_rn(lo, e1);
}

// rsqrt(mean + eps) of one row whose sum of squares the NT threads of the
// block hold as two-float partials (hi, lo): warp, then block reduction in a
// fixed order (the same result every call), the fp32 mean being the exact
// mean rounded once (unless within ~2^-40 of a rounding boundary), and a
// correctly rounded rsqrt. Every thread of the block calls it, once a kernel.
template <int NT>
__device__ __forceinline__ float block_rsqrt_mean(float hi, float lo, int H, float eps) {
    __shared__ float2 part[NT / 32];
    __shared__ float rs_s;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float h2 = __shfl_xor_sync(0xffffffffu, hi, o), l2 = __shfl_xor_sync(0xffffffffu, lo, o);
        float s1, e1;
        two_sum_f(hi, h2, s1, e1);
        hi = s1;
        lo = __fadd_rn(__fadd_rn(lo, l2), e1);
    }
    if (lane == 0) part[warp] = make_float2(hi, lo);
    __syncthreads();
    if (threadIdx.x == 0) {
        float hs = 0.f, ls = 0.f;
        for (int i = 0; i < NT / 32; ++i) {
            float s1, e1;
            two_sum_f(hs, part[i].x, s1, e1);
            hs = s1;
            ls = __fadd_rn(__fadd_rn(ls, part[i].y), e1);
        }
        // mean = (hs + ls) / H rounded once: q0 = RN(hs / H), the residual
        // hs - q0 H is exact (fma), the correction moves q0 by under half an ulp
        const float Hf = (float)H;
        const float q0 = __fdiv_rn(hs, Hf);
        const float rsd = __fadd_rn(__fmaf_rn(-q0, Hf, hs), ls);
        const float mean = __fadd_rn(q0, __fdiv_rn(rsd, Hf));
        rs_s = __frsqrt_rn(__fadd_rn(mean, eps));
    }
    __syncthreads();
    return rs_s;
}

}  // namespace moe
