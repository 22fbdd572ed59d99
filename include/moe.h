/*
 * moe.h - C ABI of the B300 (sm_103a) decode-time Mixture-of-Experts expert path.
 *
 * One token (or a small batch of tokens) through one MoE layer: RMSNorm, a
 * bf16 router matvec, softmax and top-K over the experts, for each chosen
 * expert a fused affine-dequantised (4-bit or 2-bit codes, per-group bf16
 * scale and bias) gate/up matvec with SwiGLU and a dequantised down matvec,
 * then the routing-weighted combine with an always-on shared expert and the
 * residual.  The Flash-MoE pages describe this path for Apple GPUs:
 *   - "397B MoE sur MacBook : 4,4 t/s Moteur Flash-MoE", "Techniques de
 *     rupture" items 1-4 (K active experts per layer, FMA-rewritten
 *     nibble*scale+bias dequant, fused SwiGLU, RMS norm, MoE combine);
 *   - "Flash-MoE - Dizüstünde 397 milyar parametreli modeli çalıştırma",
 *     "Model mimarisi" (512 experts, hidden 4096) and "Metal Compute
 *     Shaders" (MoE combine + residual + gate).
 *
 * Conventions for every entry point
 *   - All pointers named "device" are CUDA device pointers owned by the caller;
 *     the library never allocates, frees or keeps them.  Every device pointer
 *     must be 16-byte aligned.
 *   - `stream` is a cudaStream_t passed as void*; NULL means the legacy default
 *     stream.  Work is enqueued asynchronously; no call synchronises except
 *     moe_get_device_status.
 *   - Host-detectable errors (bad sizes, NULL or misaligned pointers, a
 *     workspace that is too small) return at once, before anything is
 *     enqueued.  A failed launch returns MOE_ERR_CUDA (moe_last_error_message()
 *     gives the CUDA error text).  Errors found on the device (a bounded wait
 *     that ran out, a non-finite activation) are recorded in the workspace
 *     status word and read with moe_get_device_status.
 *   - Calls that share a workspace must be ordered on one stream; calls on
 *     different streams need different workspaces.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef void* moe_stream_t; /* a cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* a size, pointer, alignment or flag is not valid */
  MOE_ERR_UNSUPPORTED = 2, /* valid, but outside what the kernels implement */
  MOE_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed */
  MOE_ERR_TIMEOUT = 4,     /* a device-side wait ran out of time (status word) */
  MOE_ERR_NONFINITE = 5    /* a non-finite activation was seen (status word) */
} moe_status;

/* flags of moe_dims */
#define MOE_HAS_SHARED 1      /* the layer has one always-on shared expert */
#define MOE_HAS_SHARED_GATE 2 /* the shared expert is scaled by sigmoid(shared_gate . xn) */
#define MOE_NO_FUSED 4        /* moe_layer_decode: take the multi-kernel path even for B == 1 */
#define MOE_PDL 8             /* programmatic dependent launch.  moe_layer_decode, B == 1, and
                                 moe_stack_decode: the kernel's weight prefetch overlaps the previous
                                 kernel on the stream (instead of a cooperative launch; see
                                 moe_layer_decode).  B > 1 and
                                 moe_route / moe_expert_forward: each kernel of the multi-kernel path
                                 may be scheduled while its predecessor drains and waits for it on
                                 the device (griddepcontrol.wait) before touching memory. */
#define MOE_TENSOR_CORES 16   /* moe_layer_decode and moe_expert_forward, B > 1: expert matvecs as
                                 tensor-core contractions (tcgen05, fp16 dequantised weights x fp16
                                 hi/lo activations, partial sums of 512 inputs added in fp32).
                                 Workspace sizes include the path's operand buffers when the flag
                                 is set; moe_workspace_bytes must be given the same flags. */

/* Limits of this implementation (checked on entry). */
#define MOE_MAX_TOPK 8
#define MOE_MAX_EXPERTS 1024
#define MOE_MAX_HIDDEN 8192
#define MOE_MAX_INTER 4096
#define MOE_MAX_BATCH 256
#define MOE_GROUP 64

/*
 * Layer shape.  hidden H and inter I are multiples of `group`, which must be
 * 64 (the scale/bias group along each matrix's input dimension).  `bits` is
 * the code width of the routed experts, 4 or 2.  rms_eps is the RMSNorm
 * epsilon (1e-6 in the workloads here).
 */
typedef struct {
  int32_t hidden;
  int32_t inter;
  int32_t n_experts;
  int32_t top_k;
  int32_t bits;
  int32_t group;
  float rms_eps;
  int32_t flags;
} moe_dims;

/*
 * One MoE layer, all device pointers.
 *   experts       n_experts packed blobs (moe_pack_weights), blob e at
 *                 experts + e * expert_stride; expert_stride >= the packed
 *                 size for dims.bits and a multiple of 16.
 *   shared        packed blob of the shared expert (code width shared_bits,
 *                 4 or 2), or NULL when MOE_HAS_SHARED is not set.
 *   router        bf16 [n_experts, hidden], row-major.
 *   rms_gamma     bf16 [hidden] or NULL (gamma = 1).
 *   shared_gate   bf16 [hidden], read only when MOE_HAS_SHARED_GATE is set.
 */
typedef struct {
  moe_dims d;
  const void* experts;
  size_t expert_stride;
  const void* shared;
  int32_t shared_bits;
  const uint16_t* router;
  const uint16_t* rms_gamma;
  const uint16_t* shared_gate;
} moe_layer;

/*
 * Bytes of one packed expert blob of the given code width.  Gate and up rows
 * (inter rows of `hidden` inputs) and down rows (hidden rows of `inter`
 * inputs) each hold their codes followed by one (bf16 scale, bf16 bias) pair
 * per group; a row is padded to 16 bytes.  At hidden 4096, inter 1024, 4-bit
 * this is 7,077,888 bytes: the pages' "~6.75 MB" per expert ("Techniques de
 * rupture" item 1).  Returns 0 for invalid dims or bits.
 */
size_t moe_packed_expert_bytes(const moe_dims* dims, int32_t bits);

/*
 * Bytes of device workspace the calls below need for batches of up to
 * max_batch tokens.  The workspace holds the device status word, the barrier
 * counters of the single-token fused kernel and intermediate activations.
 * Returns 0 for invalid arguments.
 */
size_t moe_workspace_bytes(const moe_dims* dims, int32_t max_batch);

/*
 * Zero a workspace (cudaMemsetAsync on `stream`).  Required once before the
 * first use of a workspace; afterwards the kernels keep it consistent.
 */
moe_status moe_workspace_init(void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * Repack one expert from the canonical layout into the blob the kernels read.
 * Canonical input, per matrix m in (gate [inter, hidden], up [inter, hidden],
 * down [hidden, inter]):
 *   codes[m]   uint8 [rows, cols*bits/8], row-major; element c of a row is
 *              bit field (c mod 8/bits) of byte c*bits/8, counted from the
 *              least significant bit (low nibble = even element);
 *   scales[m]  bf16 [rows, cols/64];  biases[m] bf16 [rows, cols/64];
 *   weight     W[r][c] = code * scale[r][c/64] + bias[r][c/64]
 *              (the pages' affine dequantisation, "Techniques de rupture" item 2).
 * dst receives moe_packed_expert_bytes(dims, bits) bytes.  Device pointers;
 * code rows must start 16-byte aligned (cols*bits/8 a multiple of 16).
 */
moe_status moe_pack_weights(const moe_dims* dims, int32_t bits,
                            const uint8_t* const codes[3],
                            const uint16_t* const scales[3],
                            const uint16_t* const biases[3],
                            void* dst, moe_stream_t stream);

/*
 * Routing of B tokens (device pointers):
 *   logits[b][e] = router[e] . xn[b] (+ logit_offset[b][e])  (fp32 accumulate)
 *   idx[b][0..K)  the K experts with the largest logits, by (logit desc,
 *                 index asc);  w[b][k] = softmax(logits[b])[idx] renormalised
 *                 over the K chosen (so the weights of a token sum to 1).
 * xn fp32 [B, hidden] is the normalised hidden state; logit_offset fp32
 * [B, n_experts] or NULL; idx int32 [B, K]; w fp32 [B, K]; logits_out fp32
 * [B, n_experts] or NULL.  The pages route on the CPU ("Techniques de
 * rupture" item 3, the deferred GPU pipeline); here routing stays on the device.
 */
moe_status moe_route(const moe_dims* dims, const float* xn, int32_t B,
                     const uint16_t* router, const float* logit_offset,
                     int32_t* idx, float* w, float* logits_out,
                     void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * One expert on B tokens (device pointers):
 *   g = Wg xn, u = Wu xn, a = silu(g) * u, d = Wd a   (SwiGLU expert)
 *   out[b] = (accumulate ? out[b] : 0) + row_w[b] * d[b]
 * blob is a packed expert of code width `bits`; xn fp32 [B, hidden]; row_w
 * fp32 [B] or NULL (weight 1); out fp32 [B, hidden].
 */
moe_status moe_expert_forward(const moe_dims* dims, int32_t bits, const void* blob,
                              const float* xn, int32_t B, const float* row_w,
                              float* out, int32_t accumulate,
                              void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * The whole layer on B tokens, in place on h (fp32 [B, hidden], device):
 *   xn = RMSNorm(h) * gamma;  route(xn) -> idx, w;
 *   h  = h + sum_k w_k * expert_{idx_k}(xn) + g_s * shared(xn)
 * with g_s = 1, or sigmoid(shared_gate . xn) under MOE_HAS_SHARED_GATE.
 * logit_offset fp32 [B, n_experts] or NULL is added to the router logits.
 * idx_out int32 [B, K] and w_out fp32 [B, K] receive the routing, or NULL.
 * B == 1 runs one persistent kernel, one block per SM (a cooperative launch,
 * or under MOE_PDL a programmatic dependent launch) when the shape fits it
 * (hidden <= 4096, inter <= 2048, experts <= 1024, top_k <= 8), else the
 * multi-kernel path; B > 1 groups the tokens by expert so that each touched
 * expert is streamed once per call (the shared expert first, in pieces of at
 * most 32 tokens).
 */
moe_status moe_layer_decode(const moe_layer* layer, float* h, int32_t B,
                            const float* logit_offset, int32_t* idx_out, float* w_out,
                            void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * One token through n_layers layers in order, in place on h (fp32 [hidden],
 * device): layer l applies moe_layer_decode's step (B = 1) to the output of
 * layer l - 1, so that on return h holds the last layer's output.  This is the
 * per-token layer loop of the pages' engine ("Techniques de rupture" item 3:
 * expert forward, then combine + norm, then the next layer), with the
 * per-layer submission gap that the Autoresearch page's "Optimisations
 * efficaces" removes by pre-encoding taken out by construction: the layers run
 * in one launch of the single-token kernel (up to 64 layers a launch; longer
 * stacks take several launches), each layer's router rows and shared-expert
 * rows copied while the previous layer finishes.
 *   layers        host array of n_layers layers (1 <= n_layers); every layer
 *                 has the same moe_dims and shared_bits; the layers' device
 *                 buffers are read only.
 *   logit_offset  fp32 [n_layers, n_experts] (layer l's row added to its
 *                 router logits) or NULL.
 *   idx_out       int32 [n_layers, K] and w_out fp32 [n_layers, K]: layer l's
 *                 routing, or NULL.
 * Results are those of n_layers moe_layer_decode calls (B = 1) on the same
 * workspace, bit for bit.  Shapes outside the single-token kernel (see
 * moe_layer_decode), or dims with MOE_NO_FUSED, run as those calls.
 * MOE_ERR_INVALID_ARG for mismatched dims, null or misaligned pointers, a
 * workspace smaller than moe_workspace_bytes(dims, 1); device-side errors are
 * recorded in the workspace status word as for moe_layer_decode.
 */
moe_status moe_stack_decode(const moe_layer* layers, int32_t n_layers, float* h,
                            const float* logit_offset, int32_t* idx_out, float* w_out,
                            void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * Synchronise `stream`, read the workspace status word, clear it and return
 * it (MOE_OK when no device-side error was recorded).  After a device-side
 * error the kernels of later calls return early until the status is cleared.
 * MOE_ERR_TIMEOUT: a bounded device wait ran out; MOE_ERR_NONFINITE: a
 * non-finite activation; MOE_ERR_UNSUPPORTED: the tensor-core contraction met
 * a weight outside the fp16 range or an inconsistent work list.
 */
moe_status moe_get_device_status(void* ws, moe_stream_t stream);

/*
 * The single-token layer (as moe_layer_decode with B == 1) for callers that
 * cannot allocate device memory.  This call has no counterpart on the
 * Flash-MoE pages; it exists for callers that are given their input and
 * output buffers but no way to allocate: code running inside another
 * framework's memory pool, stream-ordered pipelines that forbid allocation on
 * their hot path, and plugins that may not call cudaMalloc.  Instead of a
 * caller workspace it uses a fixed array of MOE_NOALLOC_SCRATCH_BYTES of device
 * memory owned by the library (a static __device__ symbol: every GPU that
 * loads the library holds it until the process exits).  It calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *   layer, h, logit_offset, idx_out, w_out   as in moe_layer_decode, B = 1
 *   status_out   device int32, required: receives this call's device status
 *                bits (0 ok; 1 a bounded wait ran out, as MOE_ERR_TIMEOUT; 2 a
 *                non-finite activation, as MOE_ERR_NONFINITE), copied on
 *                stream.  The caller cannot read the array itself and the next
 *                call clears the error state, so this copy is the only record
 *                of a device-side error; NULL is refused (MOE_ERR_INVALID_ARG).
 * Returns MOE_ERR_UNSUPPORTED (text in moe_last_error_message) when the layer
 * needs more scratch than the array holds ((experts + 1) + (top_k + 1) * inter
 * eight-byte words plus a 256-byte header) or falls outside the single-token
 * kernel (hidden <= 4096, inter <= 2048).
 * The array's device address is looked up on every call.  The first call on a
 * device (and the first after a device reset reloads the library's module)
 * also enqueues a clear of the whole array on `stream` before the kernel; it
 * synchronises nothing else, but it is a memset node if captured, so make that
 * first call before any stream capture.
 * Every call shares the one array and keeps its contents for the next call:
 * calls that may overlap on the GPU (different streams, or graphs replayed
 * concurrently) race and must be serialised by the caller.
 */
#define MOE_NOALLOC_SCRATCH_BYTES (192u * 1024u)
moe_status moe_layer_decode_noalloc(const moe_layer* layer, float* h, const float* logit_offset,
                                    int32_t* idx_out, float* w_out, int32_t* status_out,
                                    moe_stream_t stream);

/* Test hook (no counterpart on the pages): the next moe_layer_decode_noalloc
 * call made by this thread sets its array's test word so that every
 * cross-block wait of that launch expects a later launch's data; each block
 * then gives up after its bounded wait (1 s) and the call's status_out
 * receives the timeout bit.  No GPU fault, trap or endless wait is involved.
 * The call after that runs normally.  Returns MOE_OK. */
moe_status moe_noalloc_test_timeout_next(void);

/* Static text of a status code. */
const char* moe_status_string(moe_status s);

/* Text of the last CUDA error seen by this thread inside the library ("" if none). */
const char* moe_last_error_message(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
