// Row kernels of the dense 4-bit GeGLU MLP: SelfConditioning's gate_proj,
// up_proj and down_proj QuantizedLinears with the geglu between them, and
// the decoder layer's GegluMLP ("diffusion-gemma/model.ts",
// SelfConditioning.forward and DiffusionGemmaDecoderLayer.forwardWith).
//
// The two products run on the grouped dequant-GEMM as one expert whose
// token tiles cover all T rows. The kernels here surround them: one writes
// the GEMM's input (optionally through the pre norm) and its tile list, the
// other applies the post norm (optionally after adding the embeddings).
// One CTA of 256 threads a token row; H <= 8192.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kRowThreads = 256;
constexpr int kRowChunks = 4;  // 16-byte chunks a thread

// bf16((v * rs) [* w]) of both halves, each fp32 product rounded.
__device__ __forceinline__ uint32_t scale_bf16x2(uint32_t v, float rs, const uint32_t* w) {
    const float l = __fmul_rn(__uint_as_float(v << 16), rs), h = __fmul_rn(__uint_as_float(v & 0xFFFF0000u), rs);
    if (!w) return pack_bf16x2(l, h);
    return pack_bf16x2(__fmul_rn(l, __uint_as_float(*w << 16)), __fmul_rn(h, __uint_as_float(*w & 0xFFFF0000u)));
}

__device__ __forceinline__ uint4 scale_chunk(uint4 v, float rs, const uint16_t* w, int c) {
    if (!w)
        return make_uint4(scale_bf16x2(v.x, rs, nullptr), scale_bf16x2(v.y, rs, nullptr),
                          scale_bf16x2(v.z, rs, nullptr), scale_bf16x2(v.w, rs, nullptr));
    const uint4 pw = __ldg(reinterpret_cast<const uint4*>(w) + c);
    return make_uint4(scale_bf16x2(v.x, rs, &pw.x), scale_bf16x2(v.y, rs, &pw.y), scale_bf16x2(v.z, rs, &pw.z),
                      scale_bf16x2(v.w, rs, &pw.w));
}

// Input of the dense MLP's gate_up product. Row t: xs[t] = the row, or
// RMSNorm(row, pre_w) = bf16((x * rsqrt(mean(x^2) + eps)) * pre_w) with
// fp32 steps, stored with each 8-element block of K in the interleaved
// order (the down product then writes row t of its output). CTA 0 also
// writes the tile list: token tiles of nmax rows, all of expert 0.
__global__ void __launch_bounds__(kRowThreads)
    dense_prep_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ pre_w, float eps,
                      uint16_t* __restrict__ xs, Tile* __restrict__ tiles, int32_t* __restrict__ num_tiles, int T,
                      int H, int nmax) {
    pdl_trigger();
    pdl_wait();  // the previous call's GEMMs may still read xs and the tiles
    const int t = blockIdx.x, tid = threadIdx.x, chunks = H / 8;
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H);
    uint4* dst = reinterpret_cast<uint4*>(xs + (size_t)t * H);
    uint4 v[kRowChunks];
    float hi = 0.f, lo = 0.f;
#pragma unroll
    for (int q = 0; q < kRowChunks; ++q) {
        const int c = tid + q * kRowThreads;
        v[q] = make_uint4(0, 0, 0, 0);
        if (c >= chunks) continue;
        v[q] = __ldg(src + c);
        if (pre_w) {
            sumsq_bf16x2(v[q].x, hi, lo);
            sumsq_bf16x2(v[q].y, hi, lo);
            sumsq_bf16x2(v[q].z, hi, lo);
            sumsq_bf16x2(v[q].w, hi, lo);
        }
    }
    if (pre_w) {  // uniform over the block
        const float rs = block_rsqrt_mean<kRowThreads>(hi, lo, H, eps);
#pragma unroll
        for (int q = 0; q < kRowChunks; ++q) {
            const int c = tid + q * kRowThreads;
            if (c < chunks) v[q] = scale_chunk(v[q], rs, pre_w, c);
        }
    }
#pragma unroll
    for (int q = 0; q < kRowChunks; ++q) {
        const int c = tid + q * kRowThreads;
        if (c < chunks) dst[c] = interleave8(v[q]);
    }
    if (t == 0) {
        const int ntiles = (T + nmax - 1) / nmax;
        for (int i = tid; i < ntiles; i += kRowThreads) tiles[i] = Tile{0, i * nmax, min(nmax, T - i * nmax), 0};
        if (tid == 0) {
            num_tiles[0] = ntiles;
            num_tiles[1] = min(nmax, T);
        }
    }
}

// Post norm of a dense MLP output s. Row t: c = s[t], or bf16(embeds[t] +
// s[t]) (a bf16 add: the fp32 sum of two bf16 values rounds to the same
// bf16 as their exact sum), then out = bf16((c * rsqrt(mean(c^2) + eps))
// [* w]) with fp32 steps; w null is RMSNormNoScale.
__global__ void __launch_bounds__(kRowThreads)
    add_norm_kernel(const uint16_t* __restrict__ embeds, const uint16_t* __restrict__ s,
                    const uint16_t* __restrict__ w, float eps, uint16_t* __restrict__ out, int H) {
    pdl_trigger();
    pdl_wait();
    const int t = blockIdx.x, tid = threadIdx.x, chunks = H / 8;
    const uint4* st = reinterpret_cast<const uint4*>(s + (size_t)t * H);
    const uint4* et = embeds ? reinterpret_cast<const uint4*>(embeds + (size_t)t * H) : nullptr;
    uint4 cv[kRowChunks];
    float hi = 0.f, lo = 0.f;
#pragma unroll
    for (int q = 0; q < kRowChunks; ++q) {
        const int c = tid + q * kRowThreads;
        cv[q] = make_uint4(0, 0, 0, 0);
        if (c >= chunks) continue;
        uint4 v = __ldg(st + c);
        if (et) {
            const uint4 e = __ldg(et + c);
            const uint32_t ev[4] = {e.x, e.y, e.z, e.w}, sv[4] = {v.x, v.y, v.z, v.w};
            uint32_t r[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                r[i] = pack_bf16x2(__fadd_rn(__uint_as_float(ev[i] << 16), __uint_as_float(sv[i] << 16)),
                                   __fadd_rn(__uint_as_float(ev[i] & 0xFFFF0000u), __uint_as_float(sv[i] & 0xFFFF0000u)));
            v = make_uint4(r[0], r[1], r[2], r[3]);
        }
        cv[q] = v;
        sumsq_bf16x2(v.x, hi, lo);
        sumsq_bf16x2(v.y, hi, lo);
        sumsq_bf16x2(v.z, hi, lo);
        sumsq_bf16x2(v.w, hi, lo);
    }
    const float rs = block_rsqrt_mean<kRowThreads>(hi, lo, H, eps);
    uint4* ot = reinterpret_cast<uint4*>(out + (size_t)t * H);
#pragma unroll
    for (int q = 0; q < kRowChunks; ++q) {
        const int c = tid + q * kRowThreads;
        if (c < chunks) ot[c] = scale_chunk(cv[q], rs, w, c);
    }
}

}  // namespace

cudaError_t launch_dense_prep(const uint16_t* x, const uint16_t* pre_w, float eps, uint16_t* xs, Tile* tiles,
                              int32_t* num_tiles, int T, int H, int nmax, cudaStream_t stream) {
    if (T <= 0 || H % 8 != 0 || H / 8 > kRowThreads * kRowChunks || nmax <= 0) return cudaErrorInvalidValue;
    return launch_pdl(dense_prep_kernel, dim3((unsigned)T), dim3(kRowThreads), 0, stream, x, pre_w, eps, xs, tiles,
                      num_tiles, T, H, nmax);
}

cudaError_t launch_add_norm(const uint16_t* embeds, const uint16_t* s, const uint16_t* w, float eps, uint16_t* out,
                            int T, int H, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    if (H % 8 != 0 || H / 8 > kRowThreads * kRowChunks) return cudaErrorInvalidValue;
    return launch_pdl(add_norm_kernel, dim3((unsigned)T), dim3(kRowThreads), 0, stream, embeds, s, w, eps, out, H);
}

}  // namespace moe
