/*
 * sdpa.h -- C ABI of the GB300 (sm_103a) scaled dot-product attention
 * forward pass.
 *
 * Operation.  Codelab "Attention on GPU (cuDNN and TransformerEngine)",
 * section 1 ("How attention works"):
 *
 *     O = softmax(Q K^T * scale [+ causal mask]) V
 *
 * computed per (batch, query head) in one fused kernel that never writes the
 * Sq x Skv weight matrix to memory (section 8, "Run benchmarks", sequence
 * sweep: fused kernels tile the computation instead of materialising it).
 *
 * Layout (section 3, "Create Q, K and V test arrays": (B, T, N, H)), all
 * contiguous, head dimension innermost:
 *     Q, O : [B][Sq][Hq][D]
 *     K, V : [B][Skv][Hkv][D]
 * Heads (section 9, "Compare MHA, GQA and MQA"): Hkv divides Hq and query
 * head hq reads KV head hq / (Hq / Hkv) -- MHA (Hkv = Hq), GQA, MQA (Hkv = 1).
 * Causal (section 7, "Add causal masking"): the lower triangle of the
 * Sq x Skv score matrix is kept, i.e. query row i sees keys 0..i (top-left
 * aligned when Sq != Skv; rows i >= Skv see every key).
 *
 * Ownership and execution.  The caller owns every buffer; all of Q, K, V and
 * O are device pointers (cudaMalloc / PyTorch CUDA tensors) except where a
 * function says otherwise.  The library allocates no device memory.  Work is
 * enqueued on `stream` (a cudaStream_t; NULL means the legacy default stream)
 * and the call returns without synchronising.  Every call works on the
 * calling thread's current CUDA device: the buffers and the stream must
 * belong to it.
 *
 * Errors.  Every argument is checked before any CUDA call; on a failed check
 * the function returns a status code, enqueues nothing and leaves O
 * untouched.  There is no fallback to another implementation (section 6,
 * "Force the cuDNN fused backend": an unsupported request is an error, not a
 * silent switch).  A launch failure returns SDPA_ERR_CUDA; the CUDA error is
 * available from sdpa_last_cuda_error().  A kernel that had to give up (a
 * bounded wait inside it expired) records a code in a device error word that
 * sdpa_device_error() reads.
 */
#ifndef SDPA_GB300_H
#define SDPA_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SDPA_DTYPE_BF16 = 0,   /* bfloat16 Q, K, V and O */
    SDPA_DTYPE_FP16 = 1,   /* IEEE binary16 Q, K, V and O */
    SDPA_DTYPE_E4M3 = 2    /* FP8 E4M3 Q, K, V; bfloat16 O (sdpa_fwd_fp8 only) */
} sdpa_dtype_t;

typedef enum {
    SDPA_OK = 0,
    SDPA_ERR_NULL_PTR = 1,     /* a required pointer is NULL */
    SDPA_ERR_MISALIGNED = 2,   /* a pointer is not 16-byte aligned */
    SDPA_ERR_BAD_SHAPE = 3,    /* a size is < 1 or too large */
    SDPA_ERR_HEADS = 4,        /* Hq is not a multiple of Hkv */
    SDPA_ERR_HEAD_DIM = 5,     /* D is not 32, 64 or 128 (E4M3: 64 or 128) */
    SDPA_ERR_DTYPE = 6,        /* unknown dtype, or E4M3 passed to sdpa_fwd */
    SDPA_ERR_SCALE = 7,        /* scale (or a descale) is not finite and > 0 */
    SDPA_ERR_ARCH = 8,         /* current device is not compute capability 10.3 */
    SDPA_ERR_ALIAS = 9,        /* O (or LSE) overlaps an input or each other */
    SDPA_ERR_CUDA = 10,        /* a CUDA call failed; see sdpa_last_cuda_error() */
    SDPA_ERR_LAYOUT = 11,      /* a stride is unusable (see sdpa_layout_t) */
    SDPA_ERR_WORKSPACE = 12    /* workspace too small or not 16-byte aligned */
} sdpa_status_t;

/*
 * Strides of one [B][S][H][D] tensor, in elements, for the *_ex entry points.
 * The head dimension D is always contiguous.  Contiguous BSHD (the layout of
 * sdpa_fwd) is {S*H*D, H*D, D}; BHSD, the (B, N, T, H) layout section 4
 * ("Implement attention from scratch") transposes Q, K and V into before its
 * matmuls, is {H*S*D, D, S*D}.
 * Each stride must be > 0 and a multiple of 16 bytes (8 bf16 / fp16 or 16
 * E4M3 elements), below 2^40 bytes; O's strides must not map two elements to
 * one address.
 */
typedef struct {
    long long batch;   /* elements from (b, s, h, 0) to (b + 1, s, h, 0) */
    long long seq;     /* elements from (b, s, h, 0) to (b, s + 1, h, 0) */
    long long head;    /* elements from (b, s, h, 0) to (b, s, h + 1, 0) */
} sdpa_layout_t;

/*
 * Attention forward pass, bf16 or fp16 (section 6: the fused backend takes
 * 16-bit inputs).
 *   Q, K, V   device, read only, layout above, element type `dtype`.
 *   O         device, written, [B][Sq][Hq][D], element type `dtype`; must not
 *             overlap Q, K or V.
 *   B, Hq, Hkv, Sq, Skv   >= 1, Hq % Hkv == 0.
 *   D         32, 64 or 128 (section 12, "Next steps", suggests trying 32,
 *             64 and 128).
 *   scale     finite, > 0; section 4 ("Implement attention from scratch")
 *             uses 1/sqrt(D).
 *   causal    0 = no mask, nonzero = lower-triangular mask.
 *   dtype     SDPA_DTYPE_BF16 or SDPA_DTYPE_FP16.
 *   stream    cudaStream_t to enqueue on.
 * All pointers must be 16-byte aligned.  Scores and the softmax statistics
 * are fp32; O is rounded to nearest even.
 */
sdpa_status_t sdpa_fwd(const void *Q, const void *K, const void *V, void *O,
                       int B, int Hq, int Hkv, int Sq, int Skv, int D,
                       float scale, int causal, sdpa_dtype_t dtype, void *stream);

/*
 * FP8 forward pass (section 10, "Benchmark NVIDIA TransformerEngine and FP8":
 * E4M3 for the forward pass, per-tensor scales from the absolute maximum).
 *   Q, K, V   device, E4M3 bytes; the real value of an element is
 *             code * descale_x (descale_x = amax(x) / 448 for a tensor
 *             quantised with scale 448 / amax(x)).
 *   O         device, bfloat16, [B][Sq][Hq][D].
 *   descale_q, descale_k, descale_v   finite, > 0.
 * The softmax weights P are quantised to E4M3 before P V (as P * 56 with
 * P <= 8: the running max the weights are taken against may trail the row
 * max by up to a factor 8, and 8 * 56 = 448 is the largest E4M3 value), with
 * an fp32 accumulator; O is normalised by the sum of those quantised
 * weights.  Other arguments as for sdpa_fwd.
 */
sdpa_status_t sdpa_fwd_fp8(const void *Q, const void *K, const void *V, void *O,
                           int B, int Hq, int Hkv, int Sq, int Skv, int D,
                           float scale, float descale_q, float descale_k, float descale_v,
                           int causal, void *stream);

/*
 * sdpa_fwd with explicit layouts and an optional log-sum-exp output.
 *   q_layout, k_layout, v_layout, o_layout   host pointers to the strides of
 *             Q, K, V, O (sdpa_layout_t); NULL means contiguous BSHD.
 *   LSE       device, fp32 [B][Hq][Sq] contiguous, or NULL: LSE[b][hq][i] =
 *             log(sum_j exp(s_ij)) over the keys row i sees, s_ij = scale *
 *             q_i . k_j -- the log of the softmax denominator of section 1,
 *             which a backward pass or a merge of partial results needs.
 *             4-byte aligned; must not overlap Q, K, V or O.
 * Other arguments as for sdpa_fwd; O's elements are written where o_layout
 * puts them, nothing else in its span is touched.
 */
sdpa_status_t sdpa_fwd_ex(const void *Q, const void *K, const void *V, void *O, float *LSE,
                          int B, int Hq, int Hkv, int Sq, int Skv, int D,
                          const sdpa_layout_t *q_layout, const sdpa_layout_t *k_layout,
                          const sdpa_layout_t *v_layout, const sdpa_layout_t *o_layout,
                          float scale, int causal, sdpa_dtype_t dtype, void *stream);

/*
 * sdpa_fwd_fp8 with explicit layouts and an optional log-sum-exp output
 * (arguments as for sdpa_fwd_ex and sdpa_fwd_fp8).  The LSE is that of the
 * dequantised scores, scale * descale_q * descale_k * q8_i . k8_j, with the
 * row sum taken over the E4M3-rounded weights the kernel multiplies into V.
 */
sdpa_status_t sdpa_fwd_fp8_ex(const void *Q, const void *K, const void *V, void *O, float *LSE,
                              int B, int Hq, int Hkv, int Sq, int Skv, int D,
                              const sdpa_layout_t *q_layout, const sdpa_layout_t *k_layout,
                              const sdpa_layout_t *v_layout, const sdpa_layout_t *o_layout,
                              float scale, float descale_q, float descale_k, float descale_v,
                              int causal, void *stream);

/*
 * Decode-shaped forward pass (few query rows against a long key sequence),
 * non-causal, bf16 or fp16.  Section 9 ("Compare MHA, GQA and MQA") motivates
 * GQA / MQA by the KV-cache memory of inference; here the G = Hq / Hkv query
 * heads that read one KV head are stacked into the 128 rows of a query tile
 * (row s * G + h), so each K/V tile is read once for all G heads, and the key
 * sequence may be split across units whose results are merged by their
 * log-sum-exp.
 *   G         Hq / Hkv must divide 128 (SDPA_ERR_HEADS otherwise).
 *   workspace device scratch for the split results, at least
 *             sdpa_decode_workspace_bytes(...) bytes, 16-byte aligned, not
 *             overlapping Q, K, V, O or LSE; owned by the caller, contents
 *             need no initialisation, and it must not be used by another
 *             call running at the same time.  NULL: no split (one unit per
 *             KV head and group of 256 stacked rows).
 * Other arguments as for sdpa_fwd_ex (the result is the same attention).
 */
sdpa_status_t sdpa_fwd_decode(const void *Q, const void *K, const void *V, void *O, float *LSE,
                              int B, int Hq, int Hkv, int Sq, int Skv, int D,
                              const sdpa_layout_t *q_layout, const sdpa_layout_t *k_layout,
                              const sdpa_layout_t *v_layout, const sdpa_layout_t *o_layout,
                              float scale, sdpa_dtype_t dtype, void *workspace, size_t workspace_bytes,
                              void *stream);

/*
 * sdpa_fwd_decode without a caller workspace and without allocating: the
 * split results go to a 32 MiB scratch array that the library holds in
 * device memory (one per device, part of the loaded module).  The codelab
 * has no counterpart to this entry point.  It exists for callers that cannot
 * allocate or pass a workspace: a plugin or kernel hook that receives only
 * the tensors from a host framework that owns the allocator, code that must
 * not call cudaMalloc / cudaFree because they synchronise the device (a
 * latency-bound decode loop), or a caller with no free device memory to
 * spare at that point.
 *   - Cost: the module's scratch is reserved on every device where the
 *     library is loaded, by every process that uses it, even one that never
 *     calls this function.
 *   - Set-up: the first call on a device looks up the scratch's device
 *     address (cudaGetSymbolAddress, once per device, on the current device);
 *     make that first call before any stream capture.
 *   - Plans that would need more than the scratch return SDPA_ERR_WORKSPACE
 *     (none do on a device with <= 240 SMs at D <= 128).
 *   - Nothing in the scratch has to start at zero: each call writes every
 *     slot its merge step reads.
 *   - Race: all calls on a device share the one scratch array; calls must
 *     not run at the same time (issue them on one stream, or order them).
 * Arguments as for sdpa_fwd_decode.
 */
sdpa_status_t sdpa_fwd_decode_noalloc(const void *Q, const void *K, const void *V, void *O, float *LSE,
                                      int B, int Hq, int Hkv, int Sq, int Skv, int D,
                                      const sdpa_layout_t *q_layout, const sdpa_layout_t *k_layout,
                                      const sdpa_layout_t *v_layout, const sdpa_layout_t *o_layout,
                                      float scale, sdpa_dtype_t dtype, void *stream);

/*
 * Backward pass (bf16 / fp16, contiguous BSHD, D 64 or 128): the gradients of
 * sum(dO * O) for O = sdpa_fwd(Q, K, V) with the same scale and mask -- the
 * chain rule applied to section 1's definition (P = exp(S - LSE), dV = P^T dO,
 * dP = dO V^T, Delta_i = dO_i . O_i, dS = P * (dP - Delta), dQ = scale dS K,
 * dK = scale dS^T Q); section 10 names the backward pass as what training
 * runs.
 *   Q, K, V   the forward's inputs; O its output; dO the upstream gradient
 *             (shaped and typed like O); LSE the forward's log-sum-exp
 *             (fp32 [B][Hq][Sq], from sdpa_fwd_ex).  All device, read only.
 *   dQ        device, written, like Q; dK, dV device, written, like K.
 *   workspace device scratch of at least sdpa_bwd_workspace_bytes(B, Hq,
 *             Sq, D) bytes, 16-byte aligned, needing no initialisation, not
 *             used by a concurrent call.
 * Written buffers must not overlap one another or any input.  P is rounded
 * to 16 bits before dV = P^T dO, dS before dK and dQ; accumulation is fp32.
 */
sdpa_status_t sdpa_bwd(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                       const float *LSE, void *dQ, void *dK, void *dV,
                       int B, int Hq, int Hkv, int Sq, int Skv, int D,
                       float scale, int causal, sdpa_dtype_t dtype,
                       void *workspace, size_t workspace_bytes, void *stream);

/* Workspace bytes sdpa_bwd needs (0 for invalid sizes). */
size_t sdpa_bwd_workspace_bytes(int B, int Hq, int Sq, int D);

/*
 * FP8 backward pass (section 10 of the codelab, "FP8": E4M3 tensors in the
 * forward pass, E5M2 for the backward pass), contiguous BSHD, D 64 or 128:
 * the gradients of sum(dO * O) for O = sdpa_fwd_fp8(Q, K, V), every GEMM on
 * the FP8 tensor cores with fp32 accumulation; dQ sums its per-key-tile parts
 * in a bf16 accumulator (in the workspace), whose rounding is far below that
 * of the E5M2 dS it multiplies.
 *   Q8, K8, V8  E4M3 codes (one byte each) of the forward's inputs, value =
 *               code * descale_q / descale_k / descale_v.
 *   O           the forward's bf16 output; LSE its log-sum-exp (fp32
 *               [B][Hq][Sq], from sdpa_fwd_fp8_ex).
 *   dO8         E5M2 codes of the upstream gradient, value = code * descale_do.
 *   dQ, dK, dV  bf16, written, shaped like Q and K.
 *   scale_ds    per-tensor scale of dS = P * (dP - Delta) before its E5M2
 *               rounding (dS8 = e5m2(dS * scale_ds), saturating at 57344):
 *               the delayed scale of the recipe, e.g. 57344 / amax of an
 *               earlier step.  P is rounded to E4M3 as e4m3(448 P), P <= 1.
 *   amax_ds     device float, written: max |dS| of this call (before
 *               scaling), for the next call's scale_ds; NULL: not reported.
 *   workspace   device scratch of at least sdpa_bwd_fp8_workspace_bytes(B,
 *               Hq, Sq, D) bytes (B*Sq*Hq*D*2 + B*Hq*Sq*4 + 16), 16-byte
 *               aligned, needing no initialisation, not used by a
 *               concurrent call.
 * Descales and scale_ds must be finite and > 0 (else SDPA_ERR_SCALE).
 * Written buffers must not overlap one another or any input.  Other
 * arguments and statuses as for sdpa_bwd.
 */
sdpa_status_t sdpa_bwd_fp8(const void *Q8, const void *K8, const void *V8, const void *O, const void *dO8,
                           const float *LSE, void *dQ, void *dK, void *dV,
                           int B, int Hq, int Hkv, int Sq, int Skv, int D,
                           float scale, int causal, float descale_q, float descale_k, float descale_v,
                           float descale_do, float scale_ds, float *amax_ds,
                           void *workspace, size_t workspace_bytes, void *stream);

/* Workspace bytes sdpa_bwd_fp8 needs (0 for invalid sizes). */
size_t sdpa_bwd_fp8_workspace_bytes(int B, int Hq, int Sq, int D);

/*
 * Workspace bytes sdpa_fwd_decode needs for this shape on the current device
 * (0: no split, or invalid sizes).  Initialises the library on the current
 * device on first use.
 */
size_t sdpa_decode_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Skv, int D);

/* Static, human-readable name of a status code. */
const char *sdpa_status_string(sdpa_status_t status);

/* cudaError_t (as int) of the most recent SDPA_ERR_CUDA on this thread. */
int sdpa_last_cuda_error(void);

/*
 * Reads and clears the device error word of the current device (0 = none;
 * 0x1xx / 0x2xx / 0x3xx = a bounded wait of the producer / MMA issuer /
 * softmax gave up; 0x4xx / 0x5xx = a bounded wait of the 16-bit / FP8
 * backward pass gave up).  Synchronises the device.  Returns SDPA_OK or
 * SDPA_ERR_CUDA; `code` (host pointer) receives the word.
 */
sdpa_status_t sdpa_device_error(unsigned int *code);

/* Version of this ABI (bumped on any change; 2 added the *_ex entry points, 3 the decode pass,
 * 4 the backward pass, 5 the FP8 backward pass). */
int sdpa_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SDPA_GB300_H */
