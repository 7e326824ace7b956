/*
 * gdn.h -- C ABI of libgdn, the Gated DeltaNet (GDN) linear-attention layer
 * core for NVIDIA GB300 (sm_103a).
 *
 * What the library computes.  Per token t of sequence n and value head h
 * (key/query head hk = h / (Hv/Hk), contiguous groups of value heads):
 *     g_t    = -exp(A_log[h]) * softplus(a[t,h] + dt_bias[h])
 *     beta_t = sigmoid(b[t,h])
 *     qn_t   = q[t,hk] / sqrt(sum q^2 + 1e-6),  kn_t likewise
 *     S_t    = exp(g_t) S_{t-1} + kn_t (beta_t (v_t - exp(g_t) S_{t-1}^T kn_t))^T
 *     o_t    = S_t^T qn_t / sqrt(Dk)
 * with the fp32 state S held as Dk x Dv per (sequence, value head).  These are
 * the ingredients the JevAny page lists for the chunked GDN kernel ("Add
 * opt-in fused Qwen3.5 inference kernels", section Summary: gate from A_log
 * and dt_bias, beta sigmoid, q/k L2 norm, grouped value heads, followed by a
 * fused gated RMSNorm); the state layout is the "HKV" layout of the pegainfer
 * page ("feat(qwen35): add SM120 FlashInfer GDN prefill candidate", sections
 * Summary and Correctness).  Optional epilogue (JevAny page, Summary):
 *     y_t = o_t / sqrt(mean(o_t^2) + eps) * w * silu(z_t)   over Dv, per head.
 *
 * Boundary conventions (pegainfer page, review: a stable C ABI that owns the
 * kernel, unsupported shapes handled explicitly):
 *   - Every pointer is a DEVICE pointer unless stated otherwise.  The caller
 *     owns every buffer and the stream; the library never allocates, frees,
 *     prints, aborts or traps, and issues no host<->device synchronisation in
 *     gdn_prefill / gdn_decode.
 *   - Layouts are row-major, innermost index last, densely packed (the
 *     *_strided and *_conv entry points also take token inputs as strided
 *     views, see gdn_strides_t).
 *   - bf16 tensors and fp32 state/workspace pointers must be 16-byte aligned
 *     (GDN_ERR_ALIGNMENT otherwise), except a and b (2-byte, read element by
 *     element); the workspace must be 1024-byte aligned.
 *   - Only Dk = Dv = 128, Hq == Hk and Hv % Hk == 0 are supported; anything
 *     else returns GDN_ERR_UNSUPPORTED before any launch.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream).  A launch failure returns GDN_ERR_CUDA.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    int32_t num_seqs;     /* N: packed sequences (prefill) or batch (decode) */
    int32_t total_tokens; /* T_tot = cu_seqlens[N] (prefill); == N for decode */
    int32_t hq, hk, hv;   /* query, key and value heads; hq == hk, hv % hk == 0 */
    int32_t dk, dv;       /* head dims; both must be 128 */
} gdn_shape_t;

typedef enum {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1,    /* null required pointer, negative size, aliasing */
    GDN_ERR_UNSUPPORTED = 2,    /* shape outside Dk=Dv=128, Hq==Hk, Hv%Hk==0 */
    GDN_ERR_ALIGNMENT = 3,      /* pointer not 16-byte (workspace: 1024-byte) aligned */
    GDN_ERR_CUDA = 4,           /* a CUDA runtime call or launch failed */
    GDN_ERR_DEVICE_STATUS = 5,  /* a kernel recorded an error (bounded wait ran out) */
    GDN_ERR_WORKSPACE = 6       /* workspace NULL or smaller than required */
} gdn_status_t;

/* Human-readable name of a status code; never NULL. */
const char *gdn_status_string(gdn_status_t status);

/* Bytes of device workspace gdn_prefill needs for this shape (0 for an empty
 * problem).  Depends only on num_seqs, total_tokens, hk and hv.  Host-only. */
size_t gdn_prefill_workspace_bytes(const gdn_shape_t *shape);

/*
 * gdn_prefill -- chunked (64-token) prefill over packed variable-length
 * sequences (pegainfer page, Correctness: chunked vs unchunked prefill,
 * T = 1, 2, 63, 64, 65, 127, 128 operator boundaries; varlen packing).
 *
 *   q, k        bf16 [T_tot, Hk, 128]
 *   v           bf16 [T_tot, Hv, 128]
 *   a, b        bf16 [T_tot, Hv]
 *   A_log       fp32 [Hv]
 *   dt_bias     fp32 [Hv]
 *   init_state  fp32 [N, Hv, 128(k), 128(v)], or NULL for zero initial states
 *   cu_seqlens  int32 [N+1] on the device: cu[0] = 0, non-decreasing,
 *               cu[N] = T_tot.  Empty sequences are allowed (their final
 *               state is their initial state).  Not read on the host.
 *   z           bf16 [T_tot, Hv, 128] or NULL; NULL disables the epilogue
 *   norm_w      bf16 [128] (required when z != NULL), eps its epsilon
 *   out         bf16 [T_tot, Hv, 128]; must not overlap any input
 *   final_state fp32 [N, Hv, 128, 128]; may equal init_state (in place)
 *   workspace   device scratch of at least gdn_prefill_workspace_bytes(shape)
 *               bytes, 1024-byte aligned, owned by the caller; its contents
 *               need no initialisation and are garbage afterwards.  Calls that
 *               share one workspace must be ordered on the GPU.
 * Aliasing: out, final_state and the workspace (everything the call writes)
 * must not overlap one another or any input (q, k, v, a, b, z, norm_w,
 * A_log, dt_bias, init_state, cu_seqlens; strided inputs by the bytes their
 * strides span), with one exception: final_state may be exactly init_state.
 * Any other overlap returns GDN_ERR_INVALID_ARG before any launch.
 * Returns GDN_OK once the work is enqueued.
 */
gdn_status_t gdn_prefill(const gdn_shape_t *shape,
                         const void *q, const void *k, const void *v,
                         const void *a, const void *b,
                         const float *A_log, const float *dt_bias,
                         const float *init_state, const int32_t *cu_seqlens,
                         const void *z, const void *norm_w, float eps,
                         void *out, float *final_state,
                         void *workspace, size_t workspace_bytes,
                         void *stream);

/*
 * gdn_prefill_noalloc -- the same prefill as gdn_prefill for callers that
 * cannot allocate device memory: hosts that hand a kernel only their own
 * pre-registered buffers and forbid device allocation once running (an
 * allocation synchronises the device and can fragment a pool sized at
 * start-up), or plain-C callers with no device allocator.  The paper has no
 * counterpart for this entry point.
 *
 * Arguments and results are those of gdn_prefill without the workspace: the
 * scratch lives in a fixed 64 MiB array of device memory that the library
 * holds on every GPU that loads it, until the process exits.  A shape whose
 * gdn_prefill_workspace_bytes exceeds 64 MiB returns GDN_ERR_WORKSPACE
 * before any launch.  With the workspace formula that limit is
 * ceil(T_tot/64) + N <= 14 at Hv = 32 (one sequence of up to 832 tokens,
 * fewer tokens with more sequences) and <= 9 at Hv = 48.  Nothing in the
 * array needs clearing between calls.
 * The first call on a device looks up the array's device address (with that
 * device current).  Every call on a device shares the one array, so calls
 * that may overlap on the GPU (on different streams, or from different host
 * threads) race and must be ordered by the caller.  Allocates nothing.
 */
gdn_status_t gdn_prefill_noalloc(const gdn_shape_t *shape,
                                 const void *q, const void *k, const void *v,
                                 const void *a, const void *b,
                                 const float *A_log, const float *dt_bias,
                                 const float *init_state, const int32_t *cu_seqlens,
                                 const void *z, const void *norm_w, float eps,
                                 void *out, float *final_state, void *stream);

/*
 * gdn_decode -- one token per sequence, the state updated in place (the
 * recurrent-state slots of serving, SGLang page "[Perf] Pack the Qwen3.5 GDN
 * input projection on CUDA", section Accuracy Tests: mamba slots).  Each
 * 128x128 fp32 state is read once and written once.
 *
 *   shape->total_tokens must equal shape->num_seqs (= batch B).
 *   q, k   bf16 [B, Hk, 128];  v bf16 [B, Hv, 128];  a, b bf16 [B, Hv]
 *   A_log, dt_bias fp32 [Hv]
 *   state  fp32 [B, Hv, 128, 128], read and overwritten in place
 *   z      bf16 [B, Hv, 128] or NULL (no epilogue); norm_w bf16 [128]; eps
 *   out    bf16 [B, Hv, 128]; must not overlap any input or the state
 * The state must not overlap any other input either; an overlap returns
 * GDN_ERR_INVALID_ARG before any launch.  Needs no workspace.
 */
gdn_status_t gdn_decode(const gdn_shape_t *shape,
                        const void *q, const void *k, const void *v,
                        const void *a, const void *b,
                        const float *A_log, const float *dt_bias,
                        float *state,
                        const void *z, const void *norm_w, float eps,
                        void *out, void *stream);

/*
 * gdn_decode_slots -- decode of `tokens` consecutive tokens per sequence
 * (1 <= tokens <= 8: a single step, or a short draft verified together)
 * against a pool of recurrent-state slots (SGLang page "[Perf] Pack the
 * Qwen3.5 GDN input projection on CUDA", Accuracy Tests: mamba slots).
 * Each sequence's state is read once, advanced through its tokens in order
 * by the recurrence of gdn_decode, and written back once, in place.  A draft
 * of 2..8 tokens is solved together in that one pass (the recurrence
 * unrolled over the draft), which gives the token-by-token values up to
 * fp32 rounding; one token is exactly gdn_decode.
 *
 *   shape->num_seqs = B; shape->total_tokens must equal B * tokens.
 *   q, k     bf16 [B, tokens, Hk, 128];  v bf16 [B, tokens, Hv, 128]
 *   a, b     bf16 [B, tokens, Hv]
 *   A_log, dt_bias fp32 [Hv]
 *   state_pool fp32 [num_slots, Hv, 128, 128]; sequence n uses slot
 *            state_idx[n] (int32 [B] on the device), or slot n when
 *            state_idx is NULL (then num_slots must be >= B).  A negative
 *            index skips the sequence: its outputs are zero and no state is
 *            touched.  An index >= num_slots is skipped the same way and
 *            sets the range bit of the device status word.  Sequences must
 *            name distinct slots; two sequences on one slot race.
 *   z        bf16 [B, tokens, Hv, 128] or NULL (no epilogue); norm_w, eps
 *            as gdn_decode
 *   out      bf16 [B, tokens, Hv, 128]; must not overlap any input or the pool
 *            (nor may the pool overlap any other input: GDN_ERR_INVALID_ARG)
 * gdn_decode(shape, ...) is gdn_decode_slots with tokens = 1, no index and
 * num_slots = B.
 */
gdn_status_t gdn_decode_slots(const gdn_shape_t *shape, int32_t tokens, int32_t num_slots,
                              const void *q, const void *k, const void *v,
                              const void *a, const void *b,
                              const float *A_log, const float *dt_bias,
                              float *state_pool, const int32_t *state_idx,
                              const void *z, const void *norm_w, float eps,
                              void *out, void *stream);

/*
 * Strided token inputs, for reading q, k, v, z, a and b in place from one
 * packed projection output (SGLang page "[Perf] Pack the Qwen3.5 GDN input
 * projection on CUDA": a single GEMM on the packed in_proj_qkvz and
 * in_proj_ba weights writes every token's q, k, v, z, b and a side by side;
 * 12,352 elements per token for the Qwen3.5-4B geometry).  For each tensor,
 * `token` is the distance in elements between consecutive tokens and `head`
 * between consecutive heads; a head of q, k, v or z is 128 contiguous
 * elements, a head of a or b one element.  The dense layouts of gdn_prefill
 * and gdn_decode are {Hk*128, 128} for q and k, {Hv*128, 128} for v and z and
 * {Hv, 1} for a and b.
 * Requirements (else GDN_ERR_INVALID_ARG): every stride positive; for q, k,
 * v and z both strides multiples of 8 elements (16 bytes) and head >= 128.
 * z's strides are ignored when z is NULL.
 */
typedef struct {
    int64_t token;
    int64_t head;
} gdn_stride_t;

typedef struct {
    gdn_stride_t q, k, v, z, a, b;
} gdn_strides_t;

/* gdn_prefill with strided token inputs (strides NULL: the dense layouts).
 * `out` is dense [T_tot, Hv, 128] and must not overlap the span of any input. */
gdn_status_t gdn_prefill_strided(const gdn_shape_t *shape, const gdn_strides_t *strides,
                                 const void *q, const void *k, const void *v,
                                 const void *a, const void *b,
                                 const float *A_log, const float *dt_bias,
                                 const float *init_state, const int32_t *cu_seqlens,
                                 const void *z, const void *norm_w, float eps,
                                 void *out, float *final_state,
                                 void *workspace, size_t workspace_bytes,
                                 void *stream);

/* gdn_decode_slots with strided token inputs (strides NULL: the dense
 * layouts); the token index is n * tokens + t.  `out` is dense. */
gdn_status_t gdn_decode_strided(const gdn_shape_t *shape, const gdn_strides_t *strides,
                                int32_t tokens, int32_t num_slots,
                                const void *q, const void *k, const void *v,
                                const void *a, const void *b,
                                const float *A_log, const float *dt_bias,
                                float *state_pool, const int32_t *state_idx,
                                const void *z, const void *norm_w, float eps,
                                void *out, void *stream);

/*
 * Causal conv1d + SiLU ahead of the core (the JevAny page,
 * "Add opt-in fused Qwen3.5 inference kernels", Measurements, lists
 * causal-conv1d among the path's dependencies; its definition here is a
 * reading).  Over the C = Hk*128 + Hk*128 + Hv*128 channels q | k | v of
 * each token (each head 128 contiguous channels), with K = width taps:
 *     y[t, c] = silu( sum_j weight[c][j] * x[t - (K-1) + j, c] )
 * computed in fp32, rounded to bf16; the core runs on y.  Positions before a
 * sequence's first token come from its carried state: the K-1 raw inputs
 * that preceded it, oldest first.  z is not convolved.
 *   width     1..4
 *   weight    bf16 [C][width], 16-byte aligned
 *   state_in  bf16 [rows][K-1][C], 16-byte aligned: one row per sequence for
 *             prefill (rows = N; NULL means zeros), the slot pool for decode
 *             (rows = num_slots, sequence n at its slot; required if K > 1)
 *   state_out same layout: each sequence's last K-1 raw inputs after the call
 *             (for a sequence shorter than K-1, the tail of the old state
 *             followed by its tokens; an empty sequence copies its row).
 *             NULL skips it; it may equal state_in (updated in place) or lie
 *             apart from it; decode writes only the slots it names.
 * Errors: width outside 1..4 or a NULL weight, or a NULL decode state_in with
 * K > 1 -> GDN_ERR_INVALID_ARG; misaligned pointers -> GDN_ERR_ALIGNMENT;
 * state_out partially overlapping state_in, or either overlapping an output,
 * the recurrent states or the workspace -> GDN_ERR_INVALID_ARG.
 */
typedef struct {
    int32_t width;
    const void *weight;
    const void *state_in;
    void *state_out;
} gdn_conv_t;

/* Bytes of device workspace gdn_prefill_conv needs: gdn_prefill's, plus
 * room for the conv output (total_tokens x C bf16).  Host-only. */
size_t gdn_prefill_conv_workspace_bytes(const gdn_shape_t *shape);

/* gdn_prefill_strided with the conv ahead of the core; conv == NULL is
 * gdn_prefill_strided.  The conv runs as its own pass over all tokens and
 * writes its output into the workspace, which must hold
 * gdn_prefill_conv_workspace_bytes (else GDN_ERR_WORKSPACE); the core then
 * reads it there.  That output is exactly what gdn_conv_prefill writes.  The
 * carried states are rolled once every read of the old ones has finished, so
 * state_out may be state_in.  The conv weight and states follow the aliasing
 * rule of gdn_prefill (they are inputs; state_out is written). */
gdn_status_t gdn_prefill_conv(const gdn_shape_t *shape, const gdn_strides_t *strides,
                              const gdn_conv_t *conv,
                              const void *q, const void *k, const void *v,
                              const void *a, const void *b,
                              const float *A_log, const float *dt_bias,
                              const float *init_state, const int32_t *cu_seqlens,
                              const void *z, const void *norm_w, float eps,
                              void *out, float *final_state,
                              void *workspace, size_t workspace_bytes,
                              void *stream);

/* gdn_conv_prefill -- the causal conv1d + SiLU alone over packed sequences
 * (the definition above): y bf16 [T_tot][C], dense, the rows of q | k | v
 * channels, from the raw q, k, v (strided as in gdn_prefill_strided;
 * strides NULL: dense) and the carried states conv->state_in (NULL: zeros).
 * It is the pass gdn_prefill_conv runs ahead of the core, so its values are
 * bit for bit the core's inputs there, which a caller can inspect or reuse.  conv->state_out must
 * be NULL (this entry point writes y only; GDN_ERR_INVALID_ARG otherwise);
 * y must not overlap any input.  Needs no workspace. */
gdn_status_t gdn_conv_prefill(const gdn_shape_t *shape, const gdn_strides_t *strides,
                              const gdn_conv_t *conv,
                              const void *q, const void *k, const void *v,
                              const int32_t *cu_seqlens, void *y, void *stream);

/* gdn_decode_strided with the conv ahead of the core; conv->state_in is the
 * conv-state pool, indexed like state_pool.  Skipped and out-of-pool
 * sequences leave their conv state untouched.  A state_out apart from
 * state_in (a second pool, e.g. used in turn with the first) is written by
 * the decode kernel itself; with state_out == state_in a second small kernel
 * rolls the pool in place once the decode grid has finished (the value
 * heads of a group share their q and k history). */
gdn_status_t gdn_decode_conv(const gdn_shape_t *shape, const gdn_strides_t *strides,
                             const gdn_conv_t *conv, int32_t tokens, int32_t num_slots,
                             const void *q, const void *k, const void *v,
                             const void *a, const void *b,
                             const float *A_log, const float *dt_bias,
                             float *state_pool, const int32_t *state_idx,
                             const void *z, const void *norm_w, float eps,
                             void *out, void *stream);

/* Reads and clears the device status word the kernels set.  Bits:
 *   1  a bounded wait on an mbarrier ran out (the kernel skipped the rest of
 *      its waits and exited; its results are not valid)
 *   2  malformed cu_seqlens (decreasing, or outside [0, total_tokens]): the
 *      sequence was treated as empty
 *   4  a value outside the fp16 operand range (|x| > 65504) met the prefill's
 *      tensor-core path, or a decode state index was past the pool (that
 *      sequence was skipped)
 * Synchronises the device: not for the hot path.  Returns GDN_OK,
 * GDN_ERR_DEVICE_STATUS (and the raw bits in *bits when non-NULL), or
 * GDN_ERR_CUDA. */
gdn_status_t gdn_check_device_status(uint32_t *bits);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
