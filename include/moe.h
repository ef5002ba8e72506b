/*
 * libmoe -- routed 4-bit mixture-of-experts feed-forward on GB300 (sm_103a).
 *
 * The layer is the MoE branch of the DiffusionGemma-26B-A4B decoder/encoder
 * layer ("diffusion-gemma/model.ts"): class DiffRouter picks k of E experts
 * per token, class DiffExperts runs each picked expert's fused gate_up
 * SwitchLinear, GeGLU and down SwitchLinear and sums the results with the
 * routing weights.
 *
 * Conventions for every call below:
 *  - bf16 tensors are passed as uint16_t bit patterns, row-major, contiguous.
 *  - All tensor pointers are DEVICE pointers unless the name says _host.
 *    The caller owns every buffer; the library never frees caller memory.
 *  - Every device pointer must be 16-byte aligned (MOE_ERR_ALIGN otherwise).
 *  - `stream` is a cudaStream_t (NULL = legacy default stream). All work is
 *    enqueued on it; no call synchronises the host except
 *    moe_forward_hostio, moe_timing_read and moe_device_error.
 *  - Argument errors are detected on the host before anything is enqueued
 *    and leave the outputs untouched. A launch failure returns MOE_ERR_CUDA.
 *  - Supported shapes: bits == 4, group == 64, H % 128 == 0, H <= 5504,
 *    inter % 64 == 0,
 *    1 <= k <= 32, k <= E <= 256, T >= 0 (T == 0 is a no-op).
 *  - 4-bit weights use the affine layout that the pages' quantized linears
 *    consume: w uint32 [E, N, K/8] with element K of row n in nibble K%8
 *    (bits 4*(K%8)..+3, low nibble first) of word K/8; scales and biases
 *    bf16 [E, N, K/64]; the dequantised weight is bf16(scale*q + bias) and
 *    a linear computes out = in . W^T.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Shape of one layer call. eps is the RMS-norm epsilon of the router. */
typedef struct moe_dims {
    int32_t T;      /* tokens                                   */
    int32_t H;      /* hidden size                              */
    int32_t E;      /* experts                                  */
    int32_t k;      /* experts per token (top-k)                */
    int32_t inter;  /* moe_intermediate: gate_up has 2*inter rows */
    int32_t group;  /* quantisation group along K (64)          */
    int32_t bits;   /* 4                                        */
    float eps;      /* router RMS-norm epsilon                  */
} moe_dims;

/* One 4-bit affine quantized SwitchLinear for all E experts.
 * gate_up: N = 2*inter, K = H;  down: N = H, K = inter. */
typedef struct moe_qweight {
    const uint32_t* w;       /* [E, N, K/8]  */
    const uint16_t* scales;  /* [E, N, K/64] */
    const uint16_t* biases;  /* [E, N, K/64] */
} moe_qweight;

typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_NULL = 1,         /* a required pointer is NULL               */
    MOE_ERR_SHAPE = 2,        /* sizes inconsistent or out of range        */
    MOE_ERR_ALIGN = 3,        /* a pointer is not 16-byte aligned          */
    MOE_ERR_UNSUPPORTED = 4,  /* bits/group/k/E outside the supported set  */
    MOE_ERR_WORKSPACE = 5,    /* workspace too small                       */
    MOE_ERR_CUDA = 6,         /* a CUDA call or launch failed              */
    MOE_ERR_TIMEOUT = 7,      /* a kernel gave up waiting (see moe_device_error) */
    MOE_ERR_DEVICE = 8        /* no usable GPU: needs compute capability 10.3 */
} moe_status;

/* Human-readable name of a status code. Never NULL. */
const char* moe_status_str(int status);

/* Bytes of device workspace moe_experts / moe_forward / moe_forward_hostio
 * need for these dims (0 for invalid dims). Holds the routing result, the
 * expert-sorted permutation, the gathered expert inputs, the GeGLU
 * activations and the per-slot expert outputs. */
size_t moe_workspace_bytes(const moe_dims* d);

/*
 * Router (DiffRouter.forward): x [T,H] -> indices [T,k], weights [T,k].
 *   normed = rms_norm(x, no weight, eps)   fp32 inside, bf16 out
 *   normed = bf16(normed * router_scale)   per hidden dim
 *   normed = bf16(normed * bf16(H^-0.5))
 *   scores = bf16(normed . router_w^T)     [T,E]
 *   idx    = the k largest scores, value descending, ties to the lower id
 *   w      = bf16(bf16(softmax_fp32(scores[idx])) * per_expert_scale[idx])
 * x [T,H], router_w [E,H], router_scale [H], per_expert_scale [E] (bf16);
 * idx_out int32 [T,k], w_out bf16 [T,k].
 */
int moe_route(const moe_dims* d, const uint16_t* x, const uint16_t* router_w,
              const uint16_t* router_scale, const uint16_t* per_expert_scale,
              int32_t* idx_out, uint16_t* w_out, void* stream);

/*
 * Dispatch (the sorted path of DiffExperts.forward: argsort of the flat
 * indices, its inverse, rows = order // k), as a stable counting sort of the
 * flat slots f = t*k + j by expert id:
 *   offsets[e] .. offsets[e+1]   slot range of expert e (offsets int32 [E+1])
 *   perm[p] = f                  p-th slot in expert order (int32 [T*k])
 *   inv[f]  = p                  inverse of perm (int32 [T*k])
 * idx int32 [T,k] must hold ids in [0,E); a slot with a bad id is dropped
 * (inv = -1, no row in perm or offsets) and raised in moe_device_error. Bit-exact and deterministic. For T*k > 8192 the sort runs
 * as three kernels that need 64 KB of device scratch: this call allocates it
 * once per device on first use and holds it until the process exits.
 */
int moe_dispatch(const moe_dims* d, const int32_t* idx, int32_t* perm, int32_t* offsets,
                 int32_t* inv, void* stream);

/*
 * Experts (DiffExperts.forward): x [T,H], idx [T,k], w [T,k] -> out [T,H].
 * Per slot (t, j) with expert e = idx[t,j]:
 *   z = bf16(x[t] . Wgu[e]^T)          [2*inter]
 *   m = bf16(gelu_tanh(z[:inter]) * z[inter:])
 *   y = bf16(m . Wdn[e]^T)             [H]
 * out[t] = bf16( sum_j bf16(y_{t,j} * w[t,j]) ), fp32 sum in j order.
 * x may differ from the router's input (the layer routes on the residual
 * and feeds the experts its pre-feed-forward-norm-2 output). A slot whose
 * expert id lies outside [0,E) is dropped (it adds nothing to out) and
 * raised in moe_device_error.
 * workspace: moe_workspace_bytes(d) bytes of device memory, or NULL to use
 * a grow-only buffer the library owns per device (not safe for concurrent
 * calls from several host threads). out may not alias x.
 */
int moe_experts(const moe_dims* d, const uint16_t* x, const int32_t* idx, const uint16_t* w,
                const moe_qweight* gate_up, const moe_qweight* down, uint16_t* out,
                void* workspace, size_t ws_bytes, void* stream);

/*
 * Where the routed calls that take a workspace (moe_experts, moe_forward,
 * moe_forward_q4router, moe_forward_branch, moe_forward_hostio) leave the
 * dispatch of their last call inside a caller-provided workspace, as byte
 * offsets from its start: perm and inv (int32 [T*k]) and offsets (int32
 * [E+1]) exactly as moe_dispatch defines them, computed by the kernels the
 * call itself runs; idx (int32 [T,k]) and w (bf16 [T,k]) hold the routing
 * when the call was given no idx_out / w_out. For inspection and bit-exact
 * tests of the in-call dispatch; the layout depends only on the dims.
 * Returns MOE_OK, or an error for invalid dims (the map is then untouched).
 */
typedef struct moe_workspace_map {
    size_t idx, w, perm, inv, offsets;
} moe_workspace_map;
int moe_workspace_map_of(const moe_dims* d, moe_workspace_map* map);

/*
 * moe_experts without any allocation. (The pages have no counterpart: this
 * call exists for callers of this library, not for the layer.)
 *
 * Some callers cannot let a library call cudaMalloc: their device memory is
 * fully reserved by their own allocator or pool, or they cannot afford the
 * device-wide synchronisation that cudaMalloc and cudaFree may cause inside
 * a latency-critical loop. This call computes exactly what moe_experts
 * computes (same kernels, same results), but its scratch is a fixed array of
 * MOE_NOALLOC_SCRATCH_BYTES bytes inside the library's device image, which
 * every GPU that loads the library holds until the process exits. No
 * cudaMalloc, cudaFree or allocating routine is called.
 *  - Inputs and outputs are the caller's device buffers, as for moe_experts.
 *  - Dims whose scratch (moe_workspace_bytes(d)) exceeds
 *    MOE_NOALLOC_SCRATCH_BYTES are rejected with MOE_ERR_WORKSPACE before
 *    anything is enqueued (the canvas layer, T=256, H=2816, k=8, fits).
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.
 *  - All calls on a device share the one array and it keeps the last call's
 *    contents; nothing in it needs to start at zero. Calls whose work
 *    overlaps on the GPU (other streams, other host threads) race on it:
 *    serialise them.
 */
#define MOE_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
int moe_experts_noalloc(const moe_dims* d, const uint16_t* x, const int32_t* idx, const uint16_t* w,
                        const moe_qweight* gate_up, const moe_qweight* down, uint16_t* out,
                        void* stream);

/*
 * The whole layer: moe_route on x, then moe_experts on the same x.
 * idx_out / w_out may be NULL (the routing then stays in the workspace).
 */
int moe_forward(const moe_dims* d, const uint16_t* x, const uint16_t* router_w,
                const uint16_t* router_scale, const uint16_t* per_expert_scale,
                const moe_qweight* gate_up, const moe_qweight* down, uint16_t* out,
                int32_t* idx_out, uint16_t* w_out, void* workspace, size_t ws_bytes,
                void* stream);

/*
 * The router with the pages' 4-bit projection (DiffRouter.proj is a
 * QuantizedLinear): router_q is the [E, H] weight in the affine layout above
 * (w uint32 [E, H/8], scales and biases bf16 [E, H/64]); the projection uses
 * the dequantised weight bf16(S*q + B), otherwise as moe_route. E <= 128
 * (MOE_ERR_UNSUPPORTED otherwise). moe_forward_q4router is moe_forward with
 * this router.
 */
int moe_route_q4(const moe_dims* d, const uint16_t* x, const moe_qweight* router_q,
                 const uint16_t* router_scale, const uint16_t* per_expert_scale,
                 int32_t* idx_out, uint16_t* w_out, void* stream);
int moe_forward_q4router(const moe_dims* d, const uint16_t* x, const moe_qweight* router_q,
                         const uint16_t* router_scale, const uint16_t* per_expert_scale,
                         const moe_qweight* gate_up, const moe_qweight* down, uint16_t* out,
                         int32_t* idx_out, uint16_t* w_out, void* workspace, size_t ws_bytes,
                         void* stream);

/*
 * The MoE branch of the decoder layer (DiffusionGemmaDecoderLayer.forwardWith
 * in "diffusion-gemma/model.ts"): the router reads the residual, the experts
 * read preFfNorm2(residual), and the experts' combined output goes through
 * postFfNorm2. Both norms are the layer's plain RMSNorm with the weight used
 * as it is (no 1 + weight offset):
 *   norm(v, w) = bf16((v * rsqrt(mean(v^2) + eps)) * w), fp32 steps, the
 *                fp32 mean the exact mean rounded once.
 *   idx, w      = moe_route(residual)
 *   expert_in   = norm(residual, pre_norm_w)
 *   out         = norm(experts(expert_in, idx, w), post_norm_w)
 * residual [T,H], pre_norm_w [H], post_norm_w [H], out [T,H] (bf16).
 * idx_out, w_out and expert_in_out ([T,H] bf16) may be NULL; when given they
 * receive the routing and the experts' input. The expert input is written
 * by the router kernel from the rms it computes anyway; the post norm runs
 * in the combine kernel (one CTA a token). Same launches as moe_forward.
 */
int moe_forward_branch(const moe_dims* d, const uint16_t* residual, const uint16_t* router_w,
                       const uint16_t* router_scale, const uint16_t* per_expert_scale,
                       const uint16_t* pre_norm_w, const uint16_t* post_norm_w,
                       const moe_qweight* gate_up, const moe_qweight* down, uint16_t* out,
                       int32_t* idx_out, uint16_t* w_out, uint16_t* expert_in_out,
                       void* workspace, size_t ws_bytes, void* stream);

/*
 * The dense 4-bit GeGLU MLP: SelfConditioning's gate_proj, up_proj and
 * down_proj QuantizedLinears with the compiled geglu between them
 * (SelfConditioning.forward in "diffusion-gemma/model.ts"), which is also
 * how the decoder layer's GegluMLP is read (its file is not on the pages).
 * Row by row over all T rows:
 *   gate = bf16(x . W_gate^T), up = bf16(x . W_up^T)       [I] each
 *   m    = bf16(gelu_approx(gate) * up)
 *   out  = bf16(m . W_down^T)                               [H]
 * It is the routed layer's one-expert, top-1 case and runs on the same
 * grouped GEMMs: d->E and d->k must be 1 (MOE_ERR_SHAPE otherwise) and
 * d->inter is the MLP's intermediate size I (a multiple of 64).
 *   gate_up  the [2I, H] weight in the affine layout above: rows [0, I) are
 *            gate_proj, rows [I, 2I) up_proj (a checkpoint's two linears
 *            concatenated along the output dimension, with their scales and
 *            biases likewise);
 *   down     the [H, I] down_proj weight.
 * x and out [T,H] bf16. Workspace as moe_experts (moe_workspace_bytes of
 * the same dims). 3 kernel launches: input staging, gate_up + GeGLU, down.
 */
int moe_dense_mlp(const moe_dims* d, const uint16_t* x, const moe_qweight* gate_up,
                  const moe_qweight* down, uint16_t* out, void* workspace, size_t ws_bytes,
                  void* stream);

/*
 * The decoder layer's dense branch (DiffusionGemmaDecoderLayer.forwardWith):
 *   out = norm(moe_dense_mlp(norm(h, pre_norm_w)), post_norm_w)
 * with the norm of moe_forward_branch (pre_feedforward_layernorm and
 * post_feedforward_layernorm_1). The pre norm runs in the input-staging
 * kernel; the post norm adds a fourth launch (one CTA a token).
 */
int moe_dense_branch(const moe_dims* d, const uint16_t* h, const uint16_t* pre_norm_w,
                     const uint16_t* post_norm_w, const moe_qweight* gate_up,
                     const moe_qweight* down, uint16_t* out, void* workspace, size_t ws_bytes,
                     void* stream);

/*
 * SelfConditioning.forward: with s = moe_dense_mlp(norm(signal, pre_norm_w)),
 *   c   = bf16(inputs_embeds + s)                 (a bf16 add)
 *   out = bf16(c * rsqrt(mean(c^2) + eps))        (RMSNormNoScale, fp32 steps)
 * inputs_embeds, signal, out [T,H] bf16; pre_norm_w [H]. 4 launches.
 */
int moe_self_conditioning(const moe_dims* d, const uint16_t* inputs_embeds, const uint16_t* signal,
                          const uint16_t* pre_norm_w, const moe_qweight* gate_up,
                          const moe_qweight* down, uint16_t* out, void* workspace,
                          size_t ws_bytes, void* stream);

/*
 * The tied 4-bit head with the final-logit softcap
 * (DiffusionGemmaModel.logitsFromHidden in "diffusion-gemma/model.ts"):
 *   x      = bf16(h . W^T)                  the embedding table W [vocab, H]
 *                                           as a 4-bit group-64 QuantizedLinear
 *   logits = softcap * tanh(x / softcap)    fp32 steps on the widened bf16 x
 *                                           (softcap 0: logits = x)
 * The softcap's formula is read as the usual final-logit softcapping (its
 * file is not on the pages); the model's cap is 30.
 *   d       T, H as for the layer; E = k = 1 (MOE_ERR_SHAPE otherwise);
 *           inter any valid value (it only sizes unused workspace)
 *   vocab   rows of the table, a multiple of 128 (MOE_ERR_UNSUPPORTED
 *           otherwise)
 *   h       [T,H] bf16; embed the table in the affine layout above
 *           (w uint32 [vocab, H/8], scales and biases bf16 [vocab, H/64])
 *   logits  [T, vocab] float32, written whole
 * Workspace as moe_dense_mlp. 2 launches: input staging, then the grouped
 * GEMM with one expert and the softcap in its epilogue. Timing records
 * them as "gather" and "gate_up".
 */
int moe_lm_head(const moe_dims* d, int32_t vocab, float softcap, const uint16_t* h,
                const moe_qweight* embed, float* logits, void* workspace, size_t ws_bytes,
                void* stream);

/*
 * The whole layer with HOST activations: brings x_host [T,H] to the device,
 * runs moe_forward and delivers out [T,H] to out_host, then synchronises
 * the stream. Weights and router parameters are device pointers. Pinned
 * host buffers (cudaHostAlloc, cudaHostRegister) are used through their
 * device mapping: a copy kernel reads x_host into the workspace and the
 * combine writes out_host directly. Other host buffers go through
 * cudaMemcpyAsync to and from workspace copies (slower). The stream must not
 * carry other work on these host buffers meanwhile.
 */
int moe_forward_hostio(const moe_dims* d, const uint16_t* x_host, const uint16_t* router_w,
                       const uint16_t* router_scale, const uint16_t* per_expert_scale,
                       const moe_qweight* gate_up, const moe_qweight* down, uint16_t* out_host,
                       void* workspace, size_t ws_bytes, void* stream);

/*
 * Which kernels the experts part of the routed calls (moe_experts,
 * moe_experts_noalloc, moe_forward and the calls built on it) runs when
 * tokens are few. mode 0 (the default): the tcgen05 grouped dequant-GEMM for
 * every call. mode 1: a dequant-GEMV on the CUDA cores (no tensor-core
 * padding of the few rows an expert gets) for calls with T*k <= 2*E, i.e.
 * at most two rows per expert on average, token tiles of up to 4 rows. Both
 * dequantise each weight to bf16(S*q + B) and accumulate in fp32; their
 * outputs differ only by the order of the fp32 sums. On GB300 the GEMV
 * measured about half as fast as the tensor-core path at the decode size
 * (T = 8, H = 2816, E = 128, k = 8): the exact bf16 dequantisation already
 * takes most of the issue slots, and the CUDA-core products add to them,
 * while the tensor core's products cost no issue slots. The setting is
 * process-wide; change it only between calls. Returns the previous mode, or
 * -MOE_ERR_SHAPE for a mode other than 0 or 1.
 */
int moe_set_small_t_path(int mode);

/*
 * Which router kernel moe_route, moe_forward, moe_forward_branch and
 * moe_forward_q4router run (process-wide, change only between calls).
 * mode 0 (the default): one CTA per 16 tokens over the whole hidden row
 * (dense router weight, E <= 128, H a multiple of 64 up to 4416) when the
 * cluster router would walk two or more waves of tiles (large T), the
 * cluster router otherwise; mode 1: always the cluster
 * router (8-CTA thread-block clusters splitting the hidden dimension); mode
 * 2: the row router wherever it fits. Both
 * compute the same roundings (DiffRouter.forward of "diffusion-gemma/
 * model.ts": RMSNormNoScale in fp32 with the exactly rounded mean, bf16
 * after each of the three multiplies, fp32-accumulated scores rounded to
 * bf16, top k, softmax, per-expert scale); the scores' fp32 sums run in a
 * different order, so a score can round to the neighbouring bf16 value and
 * a near-tie can pick the other expert. The 4-bit projection (moe_route_q4)
 * always runs on the cluster router. Returns the previous mode, or
 * -MOE_ERR_SHAPE for a mode other than 0, 1 or 2.
 */
int moe_set_router_path(int mode);

/*
 * Per-kernel timing. After moe_timing_enable(1), each moe_forward /
 * moe_experts call records CUDA events around each of its kernels on its
 * stream (at most 1024 calls are kept). moe_timing_read synchronises the
 * recorded events and writes, for each stage, the summed milliseconds into
 * ms[0..n) in the order: route, dispatch, gather, gate_up, down, combine,
 * and the number of calls into *calls; it then clears the record. The
 * dense calls record their input staging as "gather" and their post norm
 * as "combine".
 * Returns the number of stages written.
 */
int moe_timing_enable(int enable);
int moe_timing_read(float* ms, int n, int* calls);

/* Number of kernel launches one moe_forward call with these dims makes
 * (5: router, dispatch fused with the gather, gate_up, down, combine; 8 when
 * T*k > 8192, where dispatch runs as three kernels and the gather as its
 * own); 0 if the dims are rejected. */
int moe_launches_per_forward(const moe_dims* d);

/*
 * Device-side error word of the current device: 0 if no kernel has given
 * up waiting or dropped a bad expert id since the last read; otherwise a
 * bit set (1: a pipeline wait timed out, 2: an expert id was out of range)
 * and, with bit 1, bits 8..15 naming the first wait that timed out (a
 * diagnostic code of the grouped GEMM's pipeline, 0 if not recorded).
 * Synchronises the device, then clears the word.
 */
int moe_device_error(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H_ */
