/*
 * nvfp4moe.h - C ABI of the GB300 (sm_103a) NVFP4 weight-only MoE library.
 *
 * What the library computes
 * -------------------------
 * The decode-time feed-forward layer of a Qwen3.6-35B-A3B-style mixture of
 * experts with NVFP4 weights and bf16 activations (W4A16):
 *
 *   logits[t,e] = x[t,:] . Wg[e,:]                          (bf16 router GEMV)
 *   p[t,:]      = softmax(logits[t,:])  over all E experts
 *   ids[t,:]    = the k experts with the largest p (larger first, lower id on ties)
 *   w[t,j]      = p[t,ids[t,j]] / sum_j' p[t,ids[t,j']]      (renormalise)
 *   h           = silu(G_e x) * (U_e x),  y_e = D_e h         (SwiGLU expert)
 *   y[t,:]      = sum_j w[t,j] y_{ids[t,j]}(x[t]) + sigmoid(gs . x[t]) * y_shared(x[t])
 *
 * Sources (page title, section):
 *   - lynn-engine tutorials index, row 06 "MoE router": softmax over all experts,
 *     then top-k, then renormalise; shared expert with a sigmoid gate.
 *   - lynn-engine tutorials index, "Qwen 3.6 35B-A3B" config block: hidden 2048,
 *     256 experts, 8 per token, shared expert with sigmoid_gate.
 *   - lynn-engine README (GitHub), P28 note: gate/up + SiLU consumes grouped
 *     packed NVFP4, per-16 scales and top-k ids and yields a [top_k, I]
 *     intermediate; P29 note: down + routing-weighted sum yields [H]; P45 note:
 *     one-call active-MoE ABI active_moe(hidden, ids, weights, gate_up*, down*).
 *   - Lynn Engine write-up (zingnex.cn), "1. native NVFP4 support": 4-bit NVFP4
 *     weights, bf16 activations, computed from the packed tensor with no bf16
 *     shadow copy; "P1 stage": packed E2M1 + FP16 per-16 scale projection.
 *
 * NVFP4 storage of one weight matrix W[N,K] (K % 32 == 0 for the kernels)
 * ----------------------------------------------------------------------
 *   packed  uint8 [N, K/2]    element 2j in the low nibble of byte j, 2j+1 high;
 *                             nibble = E2M1 code (bit 3 sign; magnitudes
 *                             0, .5, 1, 1.5, 2, 3, 4, 6)
 *   scales  [N, K/16]         one block scale per 16 consecutive K elements:
 *                             uint8 FP8-E4M3 (NVFP4_SCALE_E4M3), uint16
 *                             IEEE binary16 (NVFP4_SCALE_FP16) or fp32
 *                             (NVFP4_SCALE_FP32); or [N, K/32] uint8 E8M0, one
 *                             per 32 elements (NVFP4_SCALE_UE8M0)
 *   tensor_scale  one fp32    W[n,k] = E2M1 * block_scale * tensor_scale
 *
 * Conventions for every call
 * --------------------------
 *   - All array pointers are DEVICE pointers owned by the caller, 16-byte
 *     aligned, densely packed row-major. The library never allocates device or
 *     host memory and never synchronises the stream (except
 *     nvfp4_get_device_status, which says so).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Work is enqueued asynchronously on it.
 *   - Argument and shape checks run on the host, before anything is enqueued; a
 *     failing check returns its status and enqueues nothing.
 *   - A failed kernel launch returns NVFP4_ERR_CUDA. Errors that only the device
 *     can see (a non-finite weight during packing, a bounded device wait that
 *     ran out) are written to the status word of the workspace and read back
 *     with nvfp4_get_device_status.
 *   - Results are deterministic: the same inputs give the same bits on every
 *     run (no floating-point atomics anywhere).
 */
#ifndef NVFP4MOE_H
#define NVFP4MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define NVFP4MOE_VERSION 1

#if defined(__GNUC__)
#define NVFP4_API __attribute__((visibility("default")))
#else
#define NVFP4_API
#endif

typedef enum {
    NVFP4_OK = 0,
    NVFP4_ERR_INVALID_ARG = 1,        /* null pointer, negative size, bad enum     */
    NVFP4_ERR_UNSUPPORTED_SHAPE = 2,  /* shape outside the documented limits        */
    NVFP4_ERR_MISALIGNED = 3,         /* a pointer is not 16-byte aligned           */
    NVFP4_ERR_WORKSPACE_TOO_SMALL = 4,
    NVFP4_ERR_CUDA = 5,               /* a CUDA runtime call or launch failed       */
    NVFP4_ERR_DEVICE_TIMEOUT = 6,     /* a bounded device wait ran out (see below)  */
    NVFP4_ERR_NONFINITE_INPUT = 7,    /* nvfp4_pack met NaN or +-inf                */
    NVFP4_ERR_ARCH = 8                /* the current device is not sm_103           */
} nvfp4_status;

/* Block-scale contract of an NVFP4 matrix (the tag travels with every matrix and layer;
 * a call that cannot consume a kind refuses it, nothing is reinterpreted):
 *   E4M3   FP8-E4M3 scale per 16 elements, fp32 tensor scale  (the workload's format)
 *   FP16   IEEE binary16 scale per 16 elements, tensor scale 1 (README P1 stage)
 *   FP32   fp32 scale per 16 elements, tensor scale 1          (README P52: Lynn-native)
 *   UE8M0  power-of-two E8M0 scale 2^(b-127) per 32 elements, tensor scale 1
 *          (README P17/P18: the vendor MX layout, neutral byte 127)                   */
typedef enum {
    NVFP4_SCALE_E4M3 = 0,
    NVFP4_SCALE_FP16 = 1,
    NVFP4_SCALE_FP32 = 2,
    NVFP4_SCALE_UE8M0 = 3
} nvfp4_scale_kind;

/* One NVFP4 matrix W[N,K] (device pointers; see the storage section above). */
typedef struct {
    const uint8_t* packed;       /* [N, K/2]                                   */
    const void* scales;          /* [N, K/16] uint8 (E4M3) or uint16 (FP16)     */
    const float* tensor_scale;   /* one fp32                                    */
    int32_t N;
    int32_t K;
    int32_t kind;                /* nvfp4_scale_kind                            */
} nvfp4_weight;

/*
 * One MoE layer. Routed experts are stored grouped, gate and up concatenated:
 *   gu_packed [E, 2I, H/2]   rows 0..I-1 = gate G_e, rows I..2I-1 = up U_e
 *   gu_scales [E, 2I, H/16]
 *   gu_tscale [E, 2]         fp32 tensor scales of (G_e, U_e)
 *   dn_packed [E, H, I/2], dn_scales [E, H, I/16], dn_tscale [E]   (D_e)
 * The shared expert uses the same layout with E = 1 and Is in place of I:
 *   sh_gu_* [2Is, H/2] / [2Is, H/16] / [2];  sh_dn_* [H, Is/2] / [H, Is/16] / [1]
 *   sh_gate_w  bf16 [H]      the sigmoid gate vector gs
 * Is = 0 means "no shared expert" (all sh_* may then be NULL).
 * router_w is bf16 [E, H]. All scales of one layer have the same kind.
 */
typedef struct {
    int32_t H, E, k, I, Is;
    int32_t kind;                    /* nvfp4_scale_kind                        */
    const uint16_t* router_w;        /* bf16 [E, H]                              */
    const uint8_t* gu_packed;
    const void* gu_scales;
    const float* gu_tscale;
    const uint8_t* dn_packed;
    const void* dn_scales;
    const float* dn_tscale;
    const uint8_t* sh_gu_packed;
    const void* sh_gu_scales;
    const float* sh_gu_tscale;
    const uint8_t* sh_dn_packed;
    const void* sh_dn_scales;
    const float* sh_dn_tscale;
    const uint16_t* sh_gate_w;       /* bf16 [H]                                 */
} moe_layer_desc;

/* ------------------------------------------------------------------ limits */
#define NVFP4_MAX_TOPK 8          /* k <= 8                                    */
#define NVFP4_MAX_EXPERTS 256     /* E <= 256                                  */
#define NVFP4_MAX_GEMV_TOKENS 64  /* nvfp4_gemv_w4a16: 1 <= T <= 64            */
#define NVFP4_DECODE_MAX_TOKENS 64 /* moe_layer_forward: T <= 64 decode path,  */
                                   /* larger T takes the prefill path          */
#define NVFP4_MAX_TOKENS 65536     /* moe_layer_forward / workspace_size: T cap */

/*
 * nvfp4_pack - quantise an fp32 matrix to NVFP4.
 *   Defined by: Lynn Engine write-up, "1. native NVFP4 support" (4-bit E2M1
 *   weights) and "P1 stage" (per-16 FP16 scale); lynn-engine README, P89 note
 *   (one scale per 16 K elements, consumed exactly).
 *   w             fp32 [N, K] device, read only
 *   kind          NVFP4_SCALE_E4M3: tensor_scale = amax(|W|) / (6*448) (1 if
 *                 amax = 0), block code = E4M3_rne_satfinite((amax_b/6) /
 *                 tensor_scale). NVFP4_SCALE_FP16: tensor_scale = 1, block code
 *                 = FP16_rne_satfinite(amax_b/6). Every element becomes the E2M1
 *                 code nearest (ties to even, saturating at 6) to
 *                 w / (decoded block scale * tensor_scale); the sign of w is kept.
 *   packed        uint8 [N, K/2] device, written
 *   scales        [N, K/16] device (uint8 or uint16 by kind), written
 *   tensor_scale  one fp32 device, written
 *   workspace     >= nvfp4_pack_workspace_size() bytes device scratch; its status
 *                 word records NVFP4_ERR_NONFINITE_INPUT if W holds NaN/inf
 *                 (outputs are then unspecified).
 *   Shapes: N >= 1, K >= 16, K % 16 == 0.
 */
NVFP4_API nvfp4_status nvfp4_pack(const float* w, int32_t N, int32_t K, int32_t kind, uint8_t* packed,
                        void* scales, float* tensor_scale, void* workspace,
                        size_t workspace_bytes, void* stream);
NVFP4_API size_t nvfp4_pack_workspace_size(void);

/*
 * nvfp4_gemv_w4a16 - y[t,n] = sum_k W[n,k] * x[t,k] for 1..64 tokens.
 *   Defined by: Lynn Engine write-up, "P1 stage" (packed matvec computed from
 *   E2M1 + per-16 scale without a bf16 copy); lynn-engine README, P1-A
 *   (batched M > 1 packed projections).
 *   W   NVFP4 matrix (K % 32 == 0, 32 <= K <= 8192, 1 <= N <= 2^22), either
 *       scale kind
 *   x   bf16 [T, K] device;  y  bf16 [T, N] device (written; exact products,
 *       fp32 accumulation, one rounding to bf16)
 *   workspace  NULL (0 bytes), or >= 256 bytes of device memory zeroed with
 *       nvfp4_workspace_init: the call needs no scratch, but a bounded device
 *       wait that ran out is then recorded in its status word. Such a wait also
 *       writes quiet-NaN bf16 into the affected rows of y.
 *   Up to 8 tokens share one pass over the weights; T > 8 streams them
 *   ceil(T/8) times. The weights are requested before the kernel waits for the
 *   previous kernel on the stream (programmatic dependent launch), so they must
 *   not be written by a kernel that is still running; nvfp4_pack makes its
 *   output visible before it completes.
 */
NVFP4_API nvfp4_status nvfp4_gemv_w4a16(const nvfp4_weight* W, const uint16_t* x, int32_t T, uint16_t* y,
                              void* workspace, size_t workspace_bytes, void* stream);

/*
 * moe_route_topk - router tail: softmax over all E, top-k, renormalise, and
 * the per-expert token lists used by the grouped expert kernels.
 *   Defined by: lynn-engine tutorials index, row 06 "MoE router"; lynn-engine
 *   README, P35 note (sorted-router contract), P23 note (int32 ids once).
 *   logits          fp32 [T, E] device (read)
 *   topk_ids        int32 [T, k] device: experts by descending probability,
 *                   lower id first on exact ties
 *   topk_w          fp32 [T, k] device: renormalised weights (sum to 1)
 *   expert_offsets  int32 [E+1] device: token_list[expert_offsets[e] ..
 *                   expert_offsets[e+1]) are the entries routed to expert e
 *   token_list      int32 [T*k] device: entries t*k + j, grouped by expert in
 *                   ascending expert id, ascending t inside an expert
 *   Shapes: 1 <= T <= 65536, 1 <= k <= min(E, 8), E <= 256.
 */
NVFP4_API nvfp4_status moe_route_topk(const float* logits, int32_t T, int32_t E, int32_t k,
                            int32_t* topk_ids, float* topk_w, int32_t* expert_offsets,
                            int32_t* token_list, void* stream);

/*
 * moe_layer_forward - the whole layer for T tokens (router, routed experts,
 * shared expert, combine) in bf16 out.
 *   Defined by: lynn-engine README, P45 note (one-call active MoE), P28/P29
 *   notes (gate/up + SiLU, down + weighted sum), P46/P48 notes (the combine is
 *   non-atomic: every output row is owned by one thread block); tutorials
 *   index row 06 (router and sigmoid-gated shared expert).
 *   d             layer description (device pointers inside; the struct itself
 *                 is host memory, read during the call only)
 *   x             bf16 [T, H] device;  y  bf16 [T, H] device (written)
 *   topk_ids_out  int32 [T, k] device or NULL;  topk_w_out  fp32 [T, k] or NULL
 *   workspace     >= moe_layer_workspace_size(d, T) bytes of device scratch,
 *                 zeroed once with nvfp4_workspace_init before its first use
 *                 (it carries a barrier counter and the multi-token router's
 *                 completion counters across calls); calls that share a
 *                 workspace must be serialised on one stream.
 *   Shapes: H % 32 == 0, I % 32 == 0, Is % 32 == 0 (or Is == 0), 1 <= k <= 8,
 *   k <= E <= 256, 0 <= T <= 65536.
 *   Paths: T == 1 runs the one-launch decode kernel (H % 256 == 0, H <= 2048,
 *   k*I + Is <= 8192; otherwise the multi-token path), 2 <= T <= 64 the
 *   multi-token decode kernels: with E4M3 scales and H, I, Is multiples of 256
 *   (at most 4096) four launches on the warp-level tensor cores (f16 operands:
 *   weights expanded exactly, token rows scaled by a power of two per row so
 *   that no value overflows f16, the SwiGLU intermediate kept in fp32 between
 *   the passes), otherwise five launches on fp32 FMA. T > 64 with E4M3 scales
 *   and H, I, Is multiples of 256 runs the grouped prefill path (tcgen05
 *   tensor-core GEMMs with the weights expanded to bf16 in shared memory; the
 *   SwiGLU intermediate is rounded to bf16 there, the activation type). Other
 *   layers with T > 64 run as 64-token chunks of the multi-token path.
 */
NVFP4_API nvfp4_status moe_layer_forward(const moe_layer_desc* d, const uint16_t* x, int32_t T, uint16_t* y,
                               int32_t* topk_ids_out, float* topk_w_out, void* workspace,
                               size_t workspace_bytes, void* stream);
NVFP4_API size_t moe_layer_workspace_size(const moe_layer_desc* d, int32_t T);

/*
 * moe_layer_forward_residual - the layer inside a decoder block's residual stream, with
 * the pre-MoE norm fused in:
 *   x      = bf16( h / sqrt(mean_i h[t,i]^2 + eps) * (1 + norm_w) )   (RMSNorm, (1 + w) form)
 *   h_out  = bf16( h + moe_layer(x) )                                (one rounding)
 *   Defined by: lynn-engine tutorials index, row 01 (RMSNorm = (1.0 + weight) x x_norm)
 *   and the Qwen 3.6 config block (rms_norm (1.0 + weight) x x_norm); Lynn Engine
 *   write-up, "Fused Kernels" (fused RMSNorm) and the README's decode launch-overhead
 *   campaign (fused RMSNorm cut launches per token).
 *   norm_w        bf16 [H] device;  eps >= 0 (Qwen's value is 1e-6)
 *   h             bf16 [T, H] device, the residual stream;  h_out bf16 [T, H] device
 *                 (written; may be the same buffer as h)
 *   topk_ids_out, topk_w_out, workspace, stream: as for moe_layer_forward, with
 *   workspace >= moe_layer_residual_workspace_size(d, T) bytes (the layer's scratch,
 *   then the normalised rows), zeroed once with nvfp4_workspace_init.
 *   The single-token kernel computes the norm inside its activation staging and adds h
 *   in its output epilogue (still one launch); the other paths run one norm kernel
 *   first and add h in their combine epilogues. The norm is computed in fp32 (sum of
 *   squares in a fixed order, IEEE square root and division).
 */
NVFP4_API nvfp4_status moe_layer_forward_residual(const moe_layer_desc* d, const uint16_t* norm_w, float eps,
                                                  const uint16_t* h, int32_t T, uint16_t* h_out,
                                                  int32_t* topk_ids_out, float* topk_w_out, void* workspace,
                                                  size_t workspace_bytes, void* stream);
NVFP4_API size_t moe_layer_residual_workspace_size(const moe_layer_desc* d, int32_t T);

/*
 * moe_layer_forward_noalloc - the same layer as moe_layer_forward, for callers
 * that cannot allocate device memory where they run the layer (a host callback,
 * a plugin whose host framework owns all device allocations, a process whose
 * memory budget is fixed up front). The pages have no counterpart to this call:
 * it only changes where the scratch lives.
 *   Arguments as for moe_layer_forward, without the workspace. The scratch is a
 *   static 8 MiB device array inside this library; every GPU that loads the
 *   library keeps it reserved until the process exits. Nothing is allocated:
 *   no cudaMalloc, cudaFree or allocating library routine is called.
 *   The first call on a device looks up the array's device address with
 *   cudaGetSymbolAddress (with that device current); make that first call
 *   before any stream capture. Each call clears the part of the array it uses
 *   (an asynchronous memset on `stream`) and then runs the layer.
 *   All calls on a device share the one array: calls that can overlap on the
 *   GPU (different streams without ordering) race and must not be made.
 *   A layer whose scratch (moe_layer_workspace_size) exceeds 8 MiB is rejected
 *   with NVFP4_ERR_WORKSPACE_TOO_SMALL before anything is enqueued. A device-side
 *   wait that ran out is recorded in the array's status word: read it with
 *   nvfp4_noalloc_status before the next call, which clears the array.
 */
NVFP4_API nvfp4_status moe_layer_forward_noalloc(const moe_layer_desc* d, const uint16_t* x, int32_t T,
                                                 uint16_t* y, int32_t* topk_ids_out, float* topk_w_out,
                                                 void* stream);

/*
 * nvfp4_noalloc_status - the device status word of the static scratch array of
 * moe_layer_forward_noalloc on the current device: synchronises `stream`, then returns
 * NVFP4_OK or the status a kernel of the last noalloc call recorded there
 * (NVFP4_ERR_DEVICE_TIMEOUT when a bounded wait ran out; the call's outputs are then not
 * valid). clear != 0 resets the word to NVFP4_OK. NVFP4_ERR_CUDA when the array's
 * address or the copy fails.
 */
NVFP4_API nvfp4_status nvfp4_noalloc_status(int32_t clear, void* stream);

/*
 * nvfp4_scale_kind_of - which block-scale contract a stored NVFP4 matrix uses, from its
 * metadata alone (no tensor is read), so that a matrix is never consumed under the wrong
 * contract.
 *   Defined by: lynn-engine README, P59 note (a metadata-only NVFP4 layout classifier that
 *   tells the Lynn-native per-16 layout from vendor layouts before any tensor is loaded;
 *   every cross mis-load fails loud).
 *   N, K              the matrix shape (K % 16 == 0)
 *   scale_count       number of scale elements stored for the matrix
 *   scale_elem_bytes  bytes per scale element (1, 2 or 4)
 *   kind_out          host pointer, receives the nvfp4_scale_kind
 *   Returns NVFP4_OK, or NVFP4_ERR_INVALID_ARG when the metadata match no contract (for
 *   example a per-32 count with 2-byte elements, or a count that fits neither block size).
 *   Host only; enqueues nothing.
 */
NVFP4_API nvfp4_status nvfp4_scale_kind_of(int32_t N, int32_t K, size_t scale_count, int32_t scale_elem_bytes,
                                           int32_t* kind_out);

/* Zero a workspace (enqueued on `stream`). Needed once before first use, and
 * again after a call reported NVFP4_ERR_DEVICE_TIMEOUT or a CUDA error (a call
 * cut short can leave the completion counters of the multi-token router
 * non-zero; no wait depends on them, but the next call would route wrongly). */
NVFP4_API nvfp4_status nvfp4_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/* Synchronise `stream`, then read the device status word of `workspace`
 * (NVFP4_OK, NVFP4_ERR_NONFINITE_INPUT or NVFP4_ERR_DEVICE_TIMEOUT). With
 * clear != 0 the word is reset to NVFP4_OK afterwards. */
NVFP4_API nvfp4_status nvfp4_get_device_status(void* workspace, int32_t clear, void* stream);

/* Time limit, in nanoseconds, of every bounded device wait (0 restores the
 * default of 2 s). Tests lower it to make a wait run out on purpose; the
 * waiting blocks then record NVFP4_ERR_DEVICE_TIMEOUT and return. */
NVFP4_API void nvfp4_set_device_wait_limit(uint64_t limit_ns);

/* Which kernel runs a single-token (T = 1) layer call (process-wide, default 0).
 *   0  automatic: the persistent-grid form
 *   1  the persistent-grid form (one CTA per SM; the logits and the SwiGLU values are
 *      exchanged through global memory as tagged words)
 *   2  the cluster form where the shape allows it (I and Is in {256, 512, 1024}, E4M3 or
 *      FP16 scales, H <= 4096) and the device holds k clusters of 16, 12 or 8 CTAs at
 *      once (k clusters, one per routed slot; the logits and the slot's SwiGLU values are
 *      exchanged in distributed shared memory, the partial outputs through global
 *      memory); otherwise the persistent-grid form. On GB300 it runs with 12-CTA clusters
 *      on 96 SMs and measures slower than the grid form.
 * Both compute the same result within the layer's tolerance; neither changes the API's
 * arguments, workspace size or errors. Other values are taken as 0. */
NVFP4_API void nvfp4_set_single_token_form(int32_t form);

/* Which kernel a moe_layer_forward call of `T` tokens on layer `d` runs on the current
 * device under the current setting: 2 the cluster form, 1 the persistent-grid form,
 * 0 neither (multi-token kernels), -1 an invalid descriptor or no device. */
NVFP4_API int32_t nvfp4_single_token_form_used(const moe_layer_desc* d, int32_t T);

/* The cluster form's shape on the current device for layer `d`: 100 * cs + n, where cs
 * is the cluster size it uses (16, 12 or 8 CTAs: the largest whose layout fits and of
 * which the device holds k clusters at once) and n how many such clusters fit; 0 if the
 * layer has no cluster form here, -1 on error. */
NVFP4_API int32_t nvfp4_single_token_cluster_capacity(const moe_layer_desc* d);

NVFP4_API const char* nvfp4_status_string(nvfp4_status s);
NVFP4_API int32_t nvfp4_version(void);

#ifdef __cplusplus
}
#endif
#endif /* NVFP4MOE_H */
