/*
 * dr.h -- C ABI of the GB300 (sm_103a) gated delta rule library, libdr.so.
 *
 * The operation (page "NLP: linear attention summary", sections "DeltaNet", "Gated
 * DeltaNet" and "Kimi Delta Attention"):
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T,
 *     o_t = S_t^T q_t,
 *
 * per (batch b, head h), with the state S in R^{dk x dv}.  alpha_t is a scalar per head and
 * token (Gated DeltaNet), a dk-vector (KDA, per-channel gate) or 1 (DeltaNet).  The order
 * is decay, predict with the decayed state, write the beta-scaled residual, read after the
 * write (teaching loop `gated_delta_rule`, page "linear-attention gated-deltanet guide",
 * section 4).  The chunkwise-parallel form evaluated by dr_chunk_fwd (section 5 of the same
 * page; the WY representation and triangular solve named on the page "Transformer notes
 * (5): linear attention optimisations") reaches the same result up to rounding.
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers (cudaMalloc / torch CUDA memory) on the
 *     current device, contiguous, row-major, 16-byte aligned.  The caller owns every
 *     buffer; the library never allocates, frees or synchronises (except
 *     dr_get_device_status) and keeps no host-side state between calls.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy default
 *     stream).  A status of DR_OK means the work was validated and enqueued.
 *   - Token-major layouts, the layout a projection GEMM writes:
 *       q, k        [B, T, H, dk]    in_dtype
 *       v           [B, T, H, dv]    in_dtype
 *       beta        [B, T, H]        in_dtype, values in [0, 1] (logits under
 *                                    DR_FUSE_BETA_SIGMOID)
 *       log_alpha   [B, T, H] (DR_GATE_SCALAR) or [B, T, H, dk] (DR_GATE_CHANNEL), fp32,
 *                   values <= 0; NULL for DR_GATE_NONE
 *       out         [B, T, H, dv]    out_dtype
 *       states      [B, H, dk, dv]   fp32 (row i = key channel, column j = value channel)
 *     The decode entry point drops the T axis.
 *   - Inputs are assumed finite; log_alpha <= 0 and beta in [0, 1] are not checked.
 *   - Errors are returned before anything is enqueued: nothing is launched on a
 *     negative status.
 */
#ifndef DR_H_
#define DR_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same handle as cudaStream_t. */
typedef struct CUstream_st *dr_stream_t;

/* Storage dtypes. */
enum { DR_F32 = 0, DR_BF16 = 1 };

/* Gate kinds: no gate (DeltaNet), scalar per head and token (Gated DeltaNet),
   per key channel (KDA). */
enum { DR_GATE_NONE = 0, DR_GATE_SCALAR = 1, DR_GATE_CHANNEL = 2 };

/* Status codes. */
enum {
    DR_OK = 0,
    DR_ERR_INVALID = -1,      /* null pointer, bad size, misaligned pointer, bad enum   */
    DR_ERR_UNSUPPORTED = -2,  /* valid but not built: dk, dv not in {64, 128}, chunk    */
    DR_ERR_CUDA = -3,         /* a CUDA runtime call or launch failed                   */
    DR_ERR_TIMEOUT = -4,      /* a bounded device-side wait expired (device status)     */
    DR_ERR_WORKSPACE = -5     /* workspace missing or smaller than the query's answer   */
};

/* Problem descriptor of the chunkwise forward. */
typedef struct {
    int64_t B, T, H, dk, dv;  /* B, H >= 1; T >= 0; dk, dv in {64, 128}                */
    int32_t in_dtype;         /* DR_F32 or DR_BF16: q, k, v, beta                       */
    int32_t out_dtype;        /* DR_F32 or DR_BF16: out                                 */
    int32_t gate;             /* DR_GATE_*                                              */
    int32_t chunk;            /* chunk length C: 16, 32 or 64; 0 selects 64             */
} dr_chunk_desc;

/* Problem descriptor of one decode step. */
typedef struct {
    int64_t B, H, dk, dv;     /* B, H >= 1; dk, dv in {64, 128}                         */
    int32_t in_dtype;         /* DR_F32 or DR_BF16: q, k, v, beta                       */
    int32_t out_dtype;        /* DR_F32 or DR_BF16: out                                 */
    int32_t gate;             /* DR_GATE_*                                              */
    int32_t reserved;         /* must be 0                                              */
} dr_step_desc;

/*
 * Fused neighbours of the operation: the steps on either side of it in a Gated DeltaNet
 * layer (page "linear-attention gated-deltanet guide", section 4: the write gate beta, the
 * read-out gated by SiLU; q and k enter L2-normalised), applied inside the kernels of
 * dr_chunk_fwd_ex and dr_recurrent_step_ex, with no extra pass over memory.  OR-ed into
 * their `fuse` argument:
 *   DR_FUSE_QK_L2NORM      every q and k row (dk values) is divided by
 *                          sqrt(sum of squares + DR_L2NORM_EPS), in fp32, before use
 *   DR_FUSE_BETA_SIGMOID   `beta` holds logits (any finite value, in_dtype); the kernels
 *                          use beta = 1 / (1 + exp(-logit)) rounded to in_dtype, the
 *                          value a beta stored before the call would hold
 *   DR_FUSE_OUT_SILU_GATE  out = o * z * sigmoid(z), elementwise, with `z` laid out as
 *                          out ([B, T, H, dv], or [B, H, dv] for a step) in in_dtype
 * The state (init_state, final_state, the decode state) is never gated: only `out` is.
 */
enum { DR_FUSE_QK_L2NORM = 1, DR_FUSE_BETA_SIGMOID = 2, DR_FUSE_OUT_SILU_GATE = 4 };
#define DR_FUSE_ALL 7u
#define DR_L2NORM_EPS 1e-6f

/* Library version, (major << 16) | minor. */
int dr_version(void);

/* Bytes of device workspace dr_chunk_fwd takes for *desc on its fastest path; written to
   *bytes.  The answer depends only on the descriptor.  Returns DR_OK, DR_ERR_INVALID or
   DR_ERR_UNSUPPORTED.
   Few long chains (at most 76 for the tensor-core paths, at least 32 chunks each) are split
   into segments that run side by side; each (b, h, segment) then takes three dk x dv fp32
   states (the segment's transition dk x dk, its end state from a zero start, its start
   state).  Besides those:
     - bf16 inputs, dk = dv = 128, chunk 64, scalar or no gate: nothing for many chains; for
       chains split into segments, also 16.5 KB per (b, h, chunk): every chunk's
       triangular-solve operands (T = (I + A)^-1 of the WY form, page "Transformer notes
       (5): linear attention optimisations", KDA paragraph), formed for all chunks at once,
       and the row norms of the fused L2 norm;
     - the same with the per-channel gate: 131,584 bytes of tensor-core operands per
       (b, h, chunk);
     - every other configuration (the CUDA-core path): the fp32 operands W, Q*G, K*G_C/G
       [C][dk], U [C][dv], P [C][C] and G_C [dk] per (b, h, chunk). */
int dr_chunk_fwd_workspace_bytes(const dr_chunk_desc *desc, size_t *bytes);

/* The least workspace dr_chunk_fwd accepts for *desc; written to *bytes.  Equal to
   dr_chunk_fwd_workspace_bytes() except for the scalar / no-gate tensor-core configuration
   with chains split into segments, where a workspace below that size (but at least this
   one: the segments' states alone) selects a single kernel that solves inside each chain,
   with the same results up to rounding.  Returns as dr_chunk_fwd_workspace_bytes. */
int dr_chunk_fwd_min_workspace_bytes(const dr_chunk_desc *desc, size_t *bytes);

/*
 * Chunkwise forward over T tokens for all B x H chains.
 *
 *   init_state   NULL = zero initial state, else [B, H, dk, dv] fp32 (read only)
 *   out          [B, T, H, dv] out_dtype (written)
 *   final_state  NULL = not returned, else [B, H, dk, dv] fp32 (written); may equal
 *                init_state for an in-place carry, must not overlap it otherwise
 *   workspace    device scratch of at least dr_chunk_fwd_min_workspace_bytes() bytes
 *                (dr_chunk_fwd_workspace_bytes() for the fastest path); may be NULL when
 *                that size is 0.  Contents on entry are ignored; it must not be used by
 *                other work until this call's kernels finish on `stream`.
 *
 * The chunk length C only changes rounding, never the result's definition.  A tail chunk
 * (T not a multiple of C) is padded with identity steps (k = 0, beta = 0, log_alpha = 0),
 * which leave S unchanged; their outputs are not written.
 * Returns DR_OK, DR_ERR_INVALID, DR_ERR_UNSUPPORTED, DR_ERR_WORKSPACE or DR_ERR_CUDA.
 */
int dr_chunk_fwd(const dr_chunk_desc *desc,
                 const void *q, const void *k, const void *v,
                 const float *log_alpha, const void *beta,
                 const float *init_state, void *out, float *final_state,
                 void *workspace, size_t workspace_bytes, dr_stream_t stream);

/*
 * dr_chunk_fwd for callers holding HOST buffers (the end-to-end path): q, k, v, log_alpha,
 * beta, init_state are HOST pointers (layouts and dtypes as for dr_chunk_fwd), and so are
 * out and final_state (NULL = not returned).  The call copies the inputs host -> device,
 * runs the forward and copies the results device -> host, all enqueued behind `stream`
 * (the results are in place once `stream` has completed; the host buffers must not be
 * touched before).  The sequence is split into `pieces` time ranges of whole chunks (1 ..
 * 16, at most the number of chunks), the state carried from one to the next on the device:
 * one piece's kernels overlap the next piece's input copies and the previous piece's output
 * copies (the two directions also overlap each other).  Host buffers should be page-locked
 * (cudaHostAlloc / pinned) for the copies to be asynchronous.  `dev` is a device buffer of
 * at least dr_chunk_fwd_host_dev_bytes() bytes, 256-byte aligned, holding the staging
 * copies, the state and the workspace; it must not be used by other work until `stream`
 * completes.  Streams and events are created for the call and released behind its work.
 * Returns the statuses of dr_chunk_fwd (DR_ERR_WORKSPACE for a missing or short `dev`); on
 * DR_ERR_CUDA part of the work may have been enqueued; `stream` then still waits for all of it.
 */
int dr_chunk_fwd_host_dev_bytes(const dr_chunk_desc *desc, int pieces, size_t *bytes);
int dr_chunk_fwd_host(const dr_chunk_desc *desc, int pieces,
                      const void *q, const void *k, const void *v,
                      const float *log_alpha, const void *beta,
                      const float *init_state, void *out, float *final_state,
                      void *dev, size_t dev_bytes, dr_stream_t stream);

/*
 * dr_chunk_fwd with fused neighbours: `fuse` is an OR of DR_FUSE_* (0 makes the call
 * identical to dr_chunk_fwd); `z` is the output gate's input, [B, T, H, dv] in_dtype, read
 * only, required (non-NULL, 16-byte aligned, not overlapping `out`) when DR_FUSE_OUT_SILU_GATE
 * is set and ignored otherwise.  Every configuration dr_chunk_fwd accepts takes every flag.
 * The least workspace is dr_chunk_fwd_min_workspace_bytes() whatever the flags; the fastest
 * path with flags set may take more, dr_chunk_fwd_ex_workspace_bytes().  Returns the
 * statuses of dr_chunk_fwd; DR_ERR_INVALID also for bits outside DR_FUSE_ALL or a missing z.
 */
/* Bytes of device workspace dr_chunk_fwd_ex takes for *desc and the flags `fuse` on its
   fastest path; written to *bytes.  With fuse = 0, dr_chunk_fwd_workspace_bytes().  For bf16
   inputs, dk = dv = 128, chunk 64 and a scalar or no gate, with any flag set (and bf16
   outputs when the output gate is fused): the two-kernel path's 16 KB of triangular-solve
   operands plus 512 bytes of row norms per (b, h, chunk), and the segments' states when few
   long chains are split.  Returns DR_OK, DR_ERR_INVALID (also for bits outside DR_FUSE_ALL)
   or DR_ERR_UNSUPPORTED. */
int dr_chunk_fwd_ex_workspace_bytes(const dr_chunk_desc *desc, uint32_t fuse, size_t *bytes);

int dr_chunk_fwd_ex(const dr_chunk_desc *desc, uint32_t fuse,
                    const void *q, const void *k, const void *v,
                    const float *log_alpha, const void *beta, const void *z,
                    const float *init_state, void *out, float *final_state,
                    void *workspace, size_t workspace_bytes, dr_stream_t stream);

/*
 * One decode step for B x H chains, one token each (the loop body of the recurrence
 * once).  Streams the fp32 state through HBM once: it is read, decayed, updated and
 * written back in place.
 *
 *   q, k   [B, H, dk] in_dtype;  v [B, H, dv] in_dtype;  beta [B, H] in_dtype
 *   log_alpha  NULL (DR_GATE_NONE), [B, H] (scalar) or [B, H, dk] (channel), fp32
 *   state  [B, H, dk, dv] fp32, read and overwritten
 *   out    [B, H, dv] out_dtype (must not overlap state)
 * Returns DR_OK, DR_ERR_INVALID, DR_ERR_UNSUPPORTED or DR_ERR_CUDA.
 */
int dr_recurrent_step(const dr_step_desc *desc,
                      const void *q, const void *k, const void *v,
                      const float *log_alpha, const void *beta,
                      float *state, void *out, dr_stream_t stream);

/*
 * Backward of dr_chunk_fwd (training): the gradients of
 *     L = <d_out, out> + <d_final_state, final_state>
 * with respect to every input, for the same descriptor (any gate, dk, dv in {64, 128},
 * chunk 16, 32 or 64, fp32 or bf16), computed chunkwise with fp32 sums: the forward's
 * per-chunk operands and chunk-start states are recomputed into the workspace, a reverse
 * pass carries the state gradient from the last chunk to the first, and every chunk's
 * token gradients follow in parallel.  Products of rows run on the tensor cores as TF32
 * tiles, split into three products (fp32 accuracy) for fp32 inputs and single products
 * for bf16 inputs; the chunk-start states of bf16 problems that the tensor-core forward
 * serves come from it (bf16 operands).  Accuracy: fp32 inputs within 1e-4 of the exact
 * gradients (unit-scale values), bf16 inputs within the forward's bf16 bound.  The pages ask for chunkwise kernels for
 * training (page "linear-attention gated-deltanet guide", section 5) without printing a
 * backward; this is the derivative of the chunk form.
 *
 *   inputs         as for dr_chunk_fwd (q, k, v, log_alpha, beta, init_state)
 *   d_out          [B, T, H, dv] out_dtype
 *   d_final_state  NULL (zero) or [B, H, dk, dv] fp32
 *   dq, dk         [B, T, H, dk] in_dtype (written)
 *   dv             [B, T, H, dv] in_dtype (written)
 *   d_log_alpha    log_alpha's shape, fp32 (written); NULL exactly when gate is NONE
 *   d_beta         [B, T, H] in_dtype (written)
 *   d_init_state   NULL (not returned) or [B, H, dk, dv] fp32 (written)
 *   workspace      at least dr_chunk_bwd_workspace_bytes() (295,424 bytes per
 *                  (b, h, chunk) at dk = dv = 128, C = 64); contents on entry ignored
 * Written buffers must not overlap each other or any input.  The fused-neighbour flags
 * are not taken here.  Returns DR_OK, DR_ERR_INVALID, DR_ERR_UNSUPPORTED,
 * DR_ERR_WORKSPACE or DR_ERR_CUDA.
 */
int dr_chunk_bwd_workspace_bytes(const dr_chunk_desc *desc, size_t *bytes);
int dr_chunk_bwd(const dr_chunk_desc *desc,
                 const void *q, const void *k, const void *v,
                 const float *log_alpha, const void *beta, const float *init_state,
                 const void *d_out, const float *d_final_state,
                 void *dq, void *dk, void *dv, float *d_log_alpha, void *d_beta,
                 float *d_init_state, void *workspace, size_t workspace_bytes,
                 dr_stream_t stream);

/*
 * dr_recurrent_step with fused neighbours (flags as for dr_chunk_fwd_ex); `z` is
 * [B, H, dv] in_dtype, required when DR_FUSE_OUT_SILU_GATE is set, and must not overlap
 * `state` or `out`.  Returns the statuses of dr_recurrent_step.
 */
int dr_recurrent_step_ex(const dr_step_desc *desc, uint32_t fuse,
                         const void *q, const void *k, const void *v,
                         const float *log_alpha, const void *beta, const void *z,
                         float *state, void *out, dr_stream_t stream);

/*
 * dr_chunk_fwd without a caller-provided workspace.  The pages have no counterpart of
 * this entry point: it exists for callers that cannot allocate device memory -- code
 * whose host framework owns all device memory through a pre-reserved pool, plugin
 * interfaces whose execute callback must not allocate, latency-bound loops that cannot
 * pay cudaMalloc's implicit synchronisation.  They still pass inputs and outputs exactly
 * as for dr_chunk_fwd; the scratch comes from one static device array of
 * DR_NOALLOC_SCRATCH_BYTES that libdr.so holds on every GPU it is loaded on until exit.
 *
 *   - Problems whose dr_chunk_fwd_min_workspace_bytes() exceeds DR_NOALLOC_SCRATCH_BYTES
 *     are rejected with DR_ERR_WORKSPACE before anything is enqueued; the fastest path is
 *     taken whenever dr_chunk_fwd_workspace_bytes() fits.  At bf16 inputs,
 *     dk = dv = 128, C = 64: the tensor-core path (scalar or no gate) needs none
 *     unless few long chains are split into segments; the per-channel gate needs 131,584
 *     bytes per (b, h, chunk), so there B * H * ceil(T / 64) <= 510.  The CUDA-core path
 *     (fp32 inputs, other sizes) needs 147,968 bytes per (b, h, chunk) at dk = dv = 128,
 *     C = 64, so there B * H * ceil(T / 64) <= 453.
 *   - The first call on a device looks up the array's device address (cudaGetSymbolAddress
 *     with that device current); make that first call before any stream capture.
 *   - Every call shares the array.  Calls whose work overlaps on the GPU (other streams,
 *     other host threads) race on it; the caller must serialise them.  No contents need
 *     clearing between calls: every scratch element read is first written by the call.
 *   - Allocates nothing: no cudaMalloc, no cudaFree, no allocating library routine.
 * Returns the statuses of dr_chunk_fwd, and DR_ERR_CUDA if the address lookup fails.
 */
#define DR_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
int dr_chunk_fwd_noalloc(const dr_chunk_desc *desc,
                         const void *q, const void *k, const void *v,
                         const float *log_alpha, const void *beta,
                         const float *init_state, void *out, float *final_state,
                         dr_stream_t stream);

/* Synchronises `stream`, then returns and clears the library's sticky device status word
   on the current device (DR_OK, or DR_ERR_TIMEOUT if a bounded device wait expired), or
   DR_ERR_CUDA if the synchronisation itself failed. */
int dr_get_device_status(dr_stream_t stream);

/* Self-test of failure detection, with no GPU fault: launches one kernel whose thread waits
   on a barrier that nothing completes, with the chunk kernels' bounded-wait loop and a
   budget of `cycles` SM clock cycles (1 .. 4e9); on expiry it records DR_ERR_TIMEOUT in
   the status word that dr_get_device_status returns, and exits.  Returns DR_OK once
   enqueued, DR_ERR_INVALID for a budget out of range, DR_ERR_CUDA on a launch failure. */
int dr_selftest_bounded_wait(long long cycles, dr_stream_t stream);

/* Static, human-readable text of a status code (never NULL). */
const char *dr_strerror(int status);

#ifdef __cplusplus
}
#endif

#endif /* DR_H_ */
