/*
 * wkv.h -- C ABI of libwkv.so, the B300 (sm_103a) WKV operator of RWKV.
 *
 * The operator is the time-mixing "attention" of RWKV.  Sources, by page
 * title and section:
 *   "RWKV解读：在Transformer的时代的新RNN" (segmentfault), section
 *     "3、RWKV的网络架构": eq. (7) token shift, eq. (8) wkv and its
 *     recursive form, eq. (9) the sigmoid(r) gate;
 *   "RWKV についての調査記録" (qiita), section "wkvとは": a weighted average of
 *     v with weights from k, a bonus u for the current token, a decay growing
 *     with distance through one channel-wise vector w, channels independent;
 *     section "Trainingについて": gradients for every parameter, and time
 *     parallel training because the decay is data independent; section
 *     "RWKVとは？": in inference a token and a state go in, an output and a
 *     new state come out.
 * The pages lost every equation body; the exact form implemented is, per
 * batch row b and channel c, t in [0, T):
 *
 *   wkv_t = ( sum_{i<t} e^{-(t-1-i) w_c + k_i} v_i  +  e^{u_c + k_t} v_t )
 *         / ( sum_{i<t} e^{-(t-1-i) w_c + k_i}      +  e^{u_c + k_t}     )
 *
 * with decay w_c > 0 (passed directly; a caller holding w = exp(d) applies
 * gd = gw * w itself) and bonus u_c.
 *
 * Conventions for every entry point
 *   - Tensor arguments are DEVICE pointers owned by the caller (no host
 *     pointers).  The library allocates nothing and keeps no per-call state;
 *     all scratch lives in the caller's workspace (wkv_forward_noalloc:
 *     a fixed array in the library).  Its one device-side record is the
 *     expired-wait flag that wkv_sync_status reads.
 *   - k, v, y, gy, gk, gv are [B, T, C] row-major, C fastest.  w, u, gw, gu
 *     are [C].  Decode tensors are [L, B, C]; decode parameters [L, C].
 *   - stream is a cudaStream_t cast to void*; NULL is the legacy default
 *     stream.  Calls are asynchronous on that stream: a return of WKV_OK means
 *     the work was enqueued.
 *   - Invalid arguments are rejected on the host before anything is
 *     launched; outputs are then untouched.
 *   - Values must be finite and w >= 0; otherwise results are undefined
 *     (no device-side value checks).  Outputs must not alias inputs, except
 *     the decode state, which is updated in place.
 *   - Any element alignment is accepted; 16-byte aligned decode tensors with
 *     C % 4 == 0 take a vectorised path.
 *   - Results are bitwise reproducible for the same inputs and shapes (no
 *     floating-point atomics; gw, gu are reduced in a fixed order).
 */
#ifndef WKV_H_
#define WKV_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  WKV_OK = 0,
  WKV_ERR_INVALID_ARG = 1, /* a size <= 0, a null required pointer, an unknown dtype */
  WKV_ERR_UNSUPPORTED = 2, /* a valid request this build does not implement */
  WKV_ERR_MISALIGNED = 3,  /* reserved */
  WKV_ERR_WORKSPACE = 4,   /* workspace null or smaller than the *_workspace_bytes query */
  WKV_ERR_CUDA = 5,        /* a CUDA call failed; see wkv_last_error_string() */
  WKV_ERR_TIMEOUT = 6      /* a bounded device-side wait expired (wkv_workspace_check, wkv_sync_status) */
} wkv_status;

typedef enum { WKV_F32 = 0, WKV_BF16 = 1 } wkv_dtype;

/* Scan strategies of wkv_forward / wkv_backward (see wkv_debug_set_scan_mode). */
typedef enum { WKV_SCAN_AUTO = 0, WKV_SCAN_CHUNKED = 1, WKV_SCAN_SEQUENTIAL = 2 } wkv_scan_mode;

/* Human-readable name of a status code.  Never NULL. */
const char* wkv_status_string(int status);

/* Text of the last CUDA error seen by this thread in a wkv_* call ("" if
 * none).  Valid until the next wkv_* call on the same thread. */
const char* wkv_last_error_string(void);

/* ABI version, currently 1. */
int wkv_version(void);

/* Length in tokens of the time chunks of the chunked scans (the same for
 * every shape).  The checkpoint array of wkv_forward / wkv_backward holds
 * one state per chunk. */
int wkv_chunk_len(void);

/* Number of floats of a checkpoint array for shape (B, T, C):
 * 3 * ceil(T / wkv_chunk_len()) * B * C.  Layout [3][nchunks][B][C]: planes
 * num, den, pp of the state after each chunk (chunk j covers tokens
 * [j*Lc, min((j+1)*Lc, T)) ), so plane entry j is the state after token
 * min((j+1)*Lc, T) - 1, in the (num, den, pp) convention of
 * wkv_decode_step.  Returns 0 for invalid sizes. */
size_t wkv_checkpoint_floats(int B, int T, int C);

/* Workspace sizes in bytes (0 for invalid sizes).  A workspace must be
 * zero-filled before its first use (wkv_workspace_init, or any zeroing);
 * every call leaves it ready for the next one.  One workspace may be reused
 * by any number of calls in stream order, but not by two calls that run
 * concurrently. */
size_t wkv_forward_workspace_bytes(int B, int T, int C);
size_t wkv_backward_workspace_bytes(int B, int T, int C);

/* Zero-fills `bytes` bytes of `workspace` on `stream`. */
wkv_status wkv_workspace_init(void* workspace, size_t bytes, void* stream);

/* Synchronises `stream`, then reports whether a kernel that used this
 * workspace since the last check gave up a bounded wait (WKV_ERR_TIMEOUT;
 * its outputs are then invalid) and clears that record.  WKV_OK otherwise. */
wkv_status wkv_workspace_check(void* workspace, void* stream);

/* Synchronises `stream` (WKV_ERR_CUDA with the runtime's message if the
 * stream reports an error), then reports whether any kernel of this
 * library on the current device gave up a bounded wait since the last
 * wkv_sync_status: WKV_ERR_TIMEOUT (the outputs of that call are invalid),
 * else WKV_OK.  The record is device-wide, not per stream or workspace
 * (every workspace, and wkv_forward_noalloc's built-in scratch, feed it),
 * and taking it clears it; wkv_workspace_check keeps its own record per
 * workspace.  Call it from one host thread at a time per device. */
wkv_status wkv_sync_status(void* stream);

/*
 * wkv_forward -- the training (time-parallel) form: y[b,t,c] = wkv_t for all
 * t at once, by a chunked associative scan over T (chunk summaries combined
 * across chunks, runs and CTAs; see wkv_debug_set_scan_mode).
 *   kv_dtype  WKV_F32 (k, v are float) or WKV_BF16 (k, v are bf16); w, u, y
 *             are float in both cases and all arithmetic is fp32.
 *   ckpt      optional output (may be NULL): wkv_checkpoint_floats(B,T,C)
 *             floats receiving the state after each chunk.  Passing it to
 *             wkv_backward with the same w, k, v saves that call a pass over
 *             k and v.  The last entry is the state after the whole sequence.
 *   workspace at least wkv_forward_workspace_bytes(B, T, C) bytes.
 * Errors: WKV_ERR_INVALID_ARG (B, T or C <= 0, B*T*C >= 2^40, null w, u, k,
 * v or y, unknown kv_dtype), WKV_ERR_WORKSPACE, WKV_ERR_CUDA.
 */
wkv_status wkv_forward(int B, int T, int C, int kv_dtype, const float* w, const float* u, const void* k,
                       const void* v, float* y, float* ckpt, void* workspace, size_t workspace_bytes,
                       void* stream);

/*
 * wkv_forward_with_state -- wkv_forward continuing a sequence whose earlier
 * tokens are summarised by a carried state, and returning the state after
 * the last token: the prefill of a prompt by the time-parallel form, handed
 * to wkv_decode_step for the tokens that follow (the pages' two forms of
 * the same operator: parallel for training, recurrent for inference;
 * "RWKV解读" section "3、RWKV的网络架构": eq. (8) can be written
 * recursively; qiita "RWKVとは？": a token and a state in, an output and a
 * new state out).
 *   state_in   [3][B][C] floats, or NULL for the empty state: the planes
 *              num, den, pp of the state before token 0, in the convention
 *              of the decode step (a = num e^{pp}, b = den e^{pp} are the
 *              decayed sums over the earlier tokens; pp = -1e38 with
 *              num = den = 0 is the empty state).  The earlier tokens decay
 *              with the distance like any others.
 *   state_out  [3][B][C] floats, or NULL: the same planes after token T-1
 *              (pp the running maximum), ready for wkv_decode_step (its
 *              num, den, pp for one layer are the three planes).
 *   y          as for wkv_forward, or NULL for a state-only pass: nothing
 *              but state_out and ckpt is written (one of them must be
 *              given), and no output is read back or stored.
 *   The other arguments are those of wkv_forward; ckpt and y describe the T
 *   tokens of this call.  wkv_backward differentiates the forward pass from
 *   the empty state; wkv_backward_with_state differentiates this call,
 *   state_in included, and takes a gradient on state_out.
 * Errors: as wkv_forward (y, state_out and ckpt all NULL:
 * WKV_ERR_INVALID_ARG).
 */
wkv_status wkv_forward_with_state(int B, int T, int C, int kv_dtype, const float* w, const float* u, const void* k,
                                  const void* v, const float* state_in, float* y, float* state_out, float* ckpt,
                                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * wkv_state_fold -- the state after n consecutive segments of one sequence,
 * from each segment's own state (after its tokens, from the empty state) and
 * its length.  The decay does not depend on the data ("RWKV についての調査記録",
 * "Trainingについて"; eq. (8) written recursively, "RWKV解读" section
 * "3、RWKV的网络架构"): a segment acts on the carried state by decaying it by
 * its length and adding its own sums, a = e^{-n w} a + a_seg (b alike).  This
 * splits one long sequence over devices: each runs wkv_forward_with_state
 * with y = NULL on its segment, the [3][B][C] states are exchanged, each
 * folds the states of the segments before its own into its state_in, then
 * runs wkv_forward_with_state again for its outputs.  A state given before
 * the first segment enters as a leading segment of length 0.
 *   w        [C] device floats (the decay).
 *   states   [n][3][B][C] device floats: segment i's planes num, den, pp, as
 *            wkv_forward_with_state's state_out (the empty state, pp = -1e38
 *            with num = den = 0, for a segment without tokens).
 *   lengths  n HOST integers: segment i's tokens (>= 0), read during the call.
 *   out      [3][B][C] device floats: the state after the n segments (the
 *            empty state for n == 0).
 * Errors: WKV_ERR_INVALID_ARG (B or C <= 0, n < 0 or n > 256, a negative
 * length, w or out NULL, states or lengths NULL with n > 0), WKV_ERR_CUDA.
 */
wkv_status wkv_state_fold(int B, int C, const float* w, int n, const float* states, const long long* lengths,
                          float* out, void* stream);

/*
 * wkv_adjoint_fold -- the gradient of the start state of the first of n
 * consecutive segments of one sequence, from each segment's own start-state
 * gradient (wkv_backward_with_state with no gstate_end: what its own
 * outputs' gradients put on it) and the gradient on the last segment's end
 * state.  Through a segment of n tokens whose outputs carry no gradient the
 * adjoint of the sums only decays, la <- e^{-n w} la (lb alike), the
 * reverse of the state fold (eq. (8) written recursively, "RWKV解读" section
 * "3、RWKV的网络架构"); so the start gradient of segment i is its own plus
 * e^{-n_i w} times the start gradient of segment i + 1, folded from the last
 * segment to the first.  A sequence split along time gives each segment's
 * gstate_end this way from the later segments' summary passes.
 *   w            [C] the decay.
 *   adj          [n][3][B][C] planes (g_num, g_den, pp) per segment, in
 *                sequence order, each at its own start state's pp.
 *   lengths      [n] host array, tokens per segment (>= 0).
 *   gstate_end   [3][B][C] or NULL: the gradient on the last segment's end
 *                state, in the same planes (NULL: none).
 *   out          [3][B][C] planes of the first segment's start gradient, at
 *                its pp (gstate_end itself when n = 0).
 * Errors: WKV_ERR_INVALID_ARG (B or C <= 0, n < 0 or n > 256, a negative
 * length, w or out NULL, adj or lengths NULL with n > 0, n = 0 with no
 * gstate_end), WKV_ERR_CUDA.
 */
wkv_status wkv_adjoint_fold(int B, int C, const float* w, int n, const float* adj, const long long* lengths,
                            const float* gstate_end, float* out, void* stream);

/*
 * wkv_backward -- gradients of sum(gy * wkv) with respect to w, u, k, v.
 *   kv_dtype    WKV_F32: k, v, gy are float; WKV_BF16: k, v, gy are bf16
 *               (halving the bytes read; the arithmetic stays fp32 and
 *               gw, gu, gk, gv are float in both cases).
 *   gy          upstream gradient [B, T, C], of kv_dtype.
 *   ckpt        optional (may be NULL): the checkpoint array written by
 *               wkv_forward for the same w, k, v.  When NULL the call first
 *               recomputes it (one extra pass over k and v).
 *   gw, gu      [C] outputs, summed over b and t (overwritten, not
 *               accumulated).  gk, gv [B, T, C] outputs.
 *   workspace   at least wkv_backward_workspace_bytes(B, T, C) bytes.
 * The reverse-time adjoint recurrence is scanned in chunks from the last
 * chunk backwards; the forward states are recomputed per chunk from the
 * checkpoints.  Errors: as wkv_forward; WKV_ERR_UNSUPPORTED for WKV_BF16
 * while wkv_debug_set_scan_mode forces the chunked scan (which takes fp32
 * inputs only).
 */
wkv_status wkv_backward(int B, int T, int C, int kv_dtype, const float* w, const float* u, const void* k,
                        const void* v, const void* gy, const float* ckpt, float* gw, float* gu, float* gk,
                        float* gv, void* workspace, size_t workspace_bytes, void* stream);

/*
 * wkv_forward_gated -- the time-mixing output with its receptance gate fused
 * in ("RWKV解读" section "3、RWKV的网络架构", eq. (9): the wkv result is
 * multiplied elementwise by sigmoid of the receptance before the output
 * projection):
 *   out[b,t,c] = sigmoid(r[b,t,c]) * wkv_t,   sigmoid(r) = 1 / (1 + e^{-r}).
 * The gate is applied as each output is written: wkv itself never goes to
 * memory.
 *   r          [B, T, C] input of kv_dtype (like k and v).
 *   out        [B, T, C] float output.
 *   The other arguments (state_in, state_out, ckpt, workspace) are those of
 *   wkv_forward_with_state; ckpt serves wkv_backward_gated as it serves
 *   wkv_backward.
 * Errors: as wkv_forward (r NULL: WKV_ERR_INVALID_ARG); WKV_ERR_UNSUPPORTED
 * while wkv_debug_set_scan_mode forces the chunked scan (the gate is fused
 * into the sequential kernels only).
 */
wkv_status wkv_forward_gated(int B, int T, int C, int kv_dtype, const float* w, const float* u, const void* k,
                             const void* v, const void* r, const float* state_in, float* out, float* state_out,
                             float* ckpt, void* workspace, size_t workspace_bytes, void* stream);

/*
 * wkv_backward_gated -- gradients of sum(gout * sigmoid(r) * wkv) with
 * respect to w, u, k, v and r.  wkv_t reaches the output only through the
 * gate, so the gradient entering the recurrence is gout_t sigmoid(r_t), and
 *   gr_t = gout_t * wkv_t * sigmoid(r_t) * (1 - sigmoid(r_t)),
 * with wkv_t recomputed inside the reverse walk (the forward pass need not
 * keep it).  Both are formed as each chunk is read, from the r and gout
 * planes staged beside k and v.
 *   r, gout     [B, T, C] inputs of kv_dtype.
 *   gr          [B, T, C] float output.
 *   The other arguments are those of wkv_backward (ckpt from
 *   wkv_forward_gated or wkv_forward for the same w, k, v, or NULL;
 *   workspace at least wkv_backward_workspace_bytes(B, T, C)).
 * Errors: as wkv_backward (r or gr NULL: WKV_ERR_INVALID_ARG);
 * WKV_ERR_UNSUPPORTED while the chunked scan is forced.
 */
wkv_status wkv_backward_gated(int B, int T, int C, int kv_dtype, const float* w, const float* u, const void* k,
                              const void* v, const void* r, const void* gout, const float* ckpt, float* gw, float* gu,
                              float* gk, float* gv, float* gr, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Channel mixing's pointwise parts, forward and backward.  Channel mixing
 * computes K from the token-shifted input, V from K, and gates the result
 * with a sigmoid of its receptance ("RWKV についての調査記録", Time Mixing /
 * Channel Mixing walk-through); between the key and value projections sits
 * a squared ReLU ("Инновационная архитектура RWKV", "Механизмы
 * взаимодействия"; "RWKV解读" section "3、RWKV的网络架构", eq. (10)).  The
 * projections are the caller's matmuls; these calls are the elementwise
 * steps around them, over n contiguous floats of any shape:
 *   wkv_channel_mix_sqrelu            a   = max(k, 0)^2
 *   wkv_channel_mix_sqrelu_backward   gk  = 2 max(k, 0) ga
 *   wkv_channel_mix_gate              out = sigmoid(r) vk
 *   wkv_channel_mix_gate_backward     gvk = gout sigmoid(r),
 *                                     gr  = gout vk sigmoid(r) (1 - sigmoid(r))
 * All pointers are float device pointers of n elements; an output may be the
 * same buffer as an input (in place), other overlaps are undefined.  n == 0
 * does nothing.  Errors: WKV_ERR_INVALID_ARG (n < 0, or a pointer NULL with
 * n > 0), WKV_ERR_CUDA.
 */
wkv_status wkv_channel_mix_sqrelu(long long n, const float* k, float* a, void* stream);
wkv_status wkv_channel_mix_sqrelu_backward(long long n, const float* k, const float* ga, float* gk, void* stream);
wkv_status wkv_channel_mix_gate(long long n, const float* r, const float* vk, float* out, void* stream);
wkv_status wkv_channel_mix_gate_backward(long long n, const float* r, const float* vk, const float* gout, float* gr,
                                         float* gvk, void* stream);

/*
 * wkv_backward_with_state -- wkv_backward for a segment whose forward pass
 * started from a carried state (wkv_forward_with_state's state_in) and whose
 * end state feeds tokens after it: the gradient with respect to a carried
 * state, and the backward pass of a sequence split along time (each
 * segment's gradient at its start is the next earlier segment's gstate_end).
 *   state_in    [3][B][C] or NULL: the state the forward pass started from.
 *   gstate_end  [3][B][C] or NULL: the gradient of the loss from the tokens
 *               after the segment with respect to the state after its last
 *               token, as planes (g_num, g_den, pp): the gradient with
 *               respect to num and den of that state written at scale pp
 *               (a = num e^{pp}, so any pp near the state's own serves,
 *               e.g. state_out's pp plane, or that of the next segment's
 *               folded start state).
 *   gstate_in   [3][B][C] or NULL, output: the same planes for state_in:
 *               (g_num, g_den) with respect to state_in's num and den, and
 *               state_in's pp.  A sequence split along time passes each
 *               segment's gstate_in as the previous segment's gstate_end.
 *               The gradient with respect to pp follows as
 *               g_num num + g_den den.
 *   ckpt        as for wkv_backward, from wkv_forward_with_state with the
 *               same state_in (or NULL: recomputed from state_in).
 *   The other arguments, and gw (which then includes the decay of state_in
 *   through the segment), are those of wkv_backward.
 *   Summary pass: gk and gv both NULL (and gstate_in given) computes
 *   gstate_in alone, from gy and gstate_end, without writing anything else
 *   (gw, gu may be NULL and are not written).  It reads k, v, gy and the
 *   checkpoints once; the segments of a sequence split along time use it to
 *   exchange their start-state gradients before their full backward passes
 *   (wkv_adjoint_fold), so that those run at the same time.
 * Errors: as wkv_backward; WKV_ERR_UNSUPPORTED while the chunked scan is
 * forced.
 */
wkv_status wkv_backward_with_state(int B, int T, int C, int kv_dtype, const float* w, const float* u, const void* k,
                                   const void* v, const void* gy, const float* state_in, const float* gstate_end,
                                   const float* ckpt, float* gw, float* gu, float* gk, float* gv, float* gstate_in,
                                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * wkv_decode_step -- one RNN-mode step of L independent time-mixing layers,
 * fused: token shift (eq. 7) -> wkv from the carried state -> sigmoid(r)
 * gate (eq. 9) -> state update.  Per (l, b, c), with parameters at (l, c):
 *   xk = mu_k x + (1 - mu_k) x_prev   (xv with mu_v, xr with mu_r)
 *   wkv = (num e^{pp} + e^{u+k} v) / (den e^{pp} + e^{u+k})
 *   y = wkv / (1 + e^{-r})
 *   state <- state after token (k, v): a' = e^{-w} a + e^{k} v,
 *            b' = e^{-w} b + e^{k}, pp' = max(pp - w, k)
 * The empty state (no token yet) is num = den = 0, pp = -1e38.  The mix
 * outputs feed the caller's R, K, V projections for the next step; r, k, v
 * here are that step's projected inputs.
 *   x, x_prev, r, k, v         [L, B, C] inputs
 *   mu_k, mu_v, mu_r, w, u     [L, C] inputs
 *   num, den, pp               [L, B, C] state, read and updated in place
 *   y                          [L, B, C] output (required)
 *   xk, xv, xr                 [L, B, C] outputs, each may be NULL
 * Errors: WKV_ERR_INVALID_ARG (L, B or C <= 0, a required pointer NULL),
 * WKV_ERR_CUDA.
 */
wkv_status wkv_decode_step(int L, int B, int C, const float* x, const float* x_prev, const float* mu_k,
                           const float* mu_v, const float* mu_r, const float* r, const float* k, const float* v,
                           const float* w, const float* u, float* num, float* den, float* pp, float* y, float* xk,
                           float* xv, float* xr, void* stream);

/*
 * wkv_decode_step_bf16 -- wkv_decode_step with bf16 token inputs: x, x_prev,
 * r, k, v are [L, B, C] bf16 (the RNN mode of "RWKV についての調査記録",
 * section "RWKVとは？": a token and a state in, an output and a new state
 * out).  The parameters mu_k, mu_v, mu_r, w, u, the state num, den, pp and
 * the outputs y, xk, xv, xr stay fp32, and every operation is the fp32
 * arithmetic of wkv_decode_step on the widened inputs (a bf16 value widens
 * to fp32 exactly), so for the same rounded inputs the two calls agree bit
 * for bit.  50 bytes per element move with the mix outputs (60 with fp32
 * inputs).  Any alignment is accepted; 8-byte aligned bf16 tensors and
 * 16-byte aligned fp32 tensors with C % 4 == 0 take the vectorised path.
 * Errors: as wkv_decode_step.
 */
wkv_status wkv_decode_step_bf16(int L, int B, int C, const void* x, const void* x_prev, const float* mu_k,
                                const float* mu_v, const float* mu_r, const void* r, const void* k, const void* v,
                                const float* w, const float* u, float* num, float* den, float* pp, float* y,
                                float* xk, float* xv, float* xr, void* stream);

/*
 * wkv_token_shift -- the token shift of the training path, eq. (7) of
 * "RWKV解读" section "3、RWKV的网络架构": the input of each projection is
 * a weighted sum of the current and the previous token.  Per (b, t, c),
 * with x_{-1} = x0[b, c] (zeros when x0 is NULL):
 *     xk = mu_k x_t + (1 - mu_k) x_{t-1},  xv, xr alike with mu_v, mu_r.
 *   x                [B, T, C] input; x0 [B, C] or NULL (the token before
 *                    the sequence, e.g. the last token of the previous
 *                    segment).
 *   mu_k, mu_v, mu_r [C] mix vectors.
 *   xk, xv, xr       [B, T, C] outputs, all required (written in one pass
 *                    over x).
 * 16-byte aligned tensors with C % 4 == 0 take a vectorised path.
 * Errors: WKV_ERR_INVALID_ARG (a size <= 0, B*T*C >= 2^40, a required
 * pointer NULL), WKV_ERR_CUDA.
 */
wkv_status wkv_token_shift(int B, int T, int C, const float* x, const float* x0, const float* mu_k,
                           const float* mu_v, const float* mu_r, float* xk, float* xv, float* xr, void* stream);

/* Workspace bytes of wkv_token_shift_backward (per-slice partial sums);
 * 0 for invalid sizes. */
size_t wkv_token_shift_backward_workspace_bytes(int B, int T, int C);

/*
 * wkv_token_shift_backward -- gradients of sum(gxk xk + gxv xv + gxr xr)
 * for wkv_token_shift's inputs:
 *     gx_t  = sum_m mu_m gxm_t + (1 - mu_m) gxm_{t+1}   (no t+1 term at T-1)
 *     gx0   = sum_m (1 - mu_m) gxm_0                     [B, C], may be NULL
 *     gmu_m = sum_{b,t} gxm_t (x_t - x_{t-1})            [C]
 *   gx [B, T, C] and gmu_k, gmu_v, gmu_r [C] are required outputs
 *   (overwritten); the gmu sums are in a fixed order (bitwise reproducible).
 *   workspace  at least wkv_token_shift_backward_workspace_bytes(B, T, C)
 *              bytes of device memory (no initialisation needed).
 * Errors: as wkv_token_shift, plus WKV_ERR_WORKSPACE.
 */
wkv_status wkv_token_shift_backward(int B, int T, int C, const float* x, const float* x0, const float* mu_k,
                                    const float* mu_v, const float* mu_r, const float* gxk, const float* gxv,
                                    const float* gxr, float* gx, float* gx0, float* gmu_k, float* gmu_v,
                                    float* gmu_r, void* workspace, size_t workspace_bytes, void* stream);

/*
 * wkv_forward_noalloc -- wkv_forward without a caller-provided workspace.
 * The pages have no counterpart: this entry point exists for callers that
 * cannot call cudaMalloc, such as a plugin or embedded host whose device
 * memory belongs to another allocator, or a latency-bound loop that must
 * never allocate (cudaMalloc can synchronise the device and stall every
 * stream).  Inputs and outputs are passed exactly as for wkv_forward (y and
 * the optional ckpt are caller-owned device memory); the scratch comes from
 * one 32 MiB array compiled into the library, which every GPU that loads the
 * library holds until the process exits.  Nothing is allocated.
 *   - Shapes whose wkv_forward_workspace_bytes exceed 32 MiB are rejected
 *     with WKV_ERR_WORKSPACE and a message in wkv_last_error_string().
 *   - The array used is the current device's: make the device that holds
 *     the tensors current before the call.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - Every call on a device shares the array and it keeps the last call's
 *     contents, which the next call relies on (its tile counters are back at
 *     zero; a launch counter in it tags each call's intermediate results so
 *     that an earlier call's are never taken for the current one's).  Calls
 *     that overlap on the GPU (different streams without ordering, or
 *     different host threads) race on the array: serialise them.
 *   - A bounded device-side wait that expires is reported by
 *     wkv_sync_status (there is no workspace to check).
 * Errors: as wkv_forward, plus WKV_ERR_WORKSPACE for shapes too large.
 */
wkv_status wkv_forward_noalloc(int B, int T, int C, int kv_dtype, const float* w, const float* u, const void* k,
                               const void* v, float* y, float* ckpt, void* stream);

/*
 * Test hooks (process-wide; not for production use).
 * wkv_debug_set_wait_budget_ns: limit of each bounded device-side wait of
 *   the scans, in ns of %globaltimer; <= 0 restores the default (500 ms).
 * wkv_debug_set_skip_chunk: the results that carry time chunk `chunk` to
 *   other CTAs are never published (the chunked scan: that chunk's tiles;
 *   the sequential kernels: the summary of the run holding the chunk, when
 *   its column has several runs), so the waits of the CTAs that need them
 *   expire and the call reports WKV_ERR_TIMEOUT through
 *   wkv_workspace_check; -1 turns this off.
 */
wkv_status wkv_debug_set_wait_budget_ns(long long ns);
wkv_status wkv_debug_set_skip_chunk(int chunk);

/*
 * wkv_debug_set_scan_mode: which kernels wkv_forward and wkv_backward run
 * (process-wide; for tests and measurements).
 *   WKV_SCAN_AUTO (default): the sequential kernels, measured faster on
 *     every shape tried (from B=1 T=64 C=64 to B=1 T=131072 C=2560).
 *   WKV_SCAN_CHUNKED: time cut into 32-token chunks spread over all CTAs of
 *     a persistent launch; chunk results carried between CTAs.
 *   WKV_SCAN_SEQUENTIAL: a column (batch row, 32 channels) walks its chunks
 *     in order, split into a few runs (one warp each) that exchange one
 *     summary each.
 * Both strategies compute the same recurrence with the same per-chunk
 * arithmetic; outputs agree to rounding (bitwise, with one run per column,
 * on lanes whose chunks all stay on the fixed-scale form).
 * Errors: WKV_ERR_INVALID_ARG for another value.
 */
wkv_status wkv_debug_set_scan_mode(int mode);

/*
 * wkv_debug_set_max_runs: upper bound on the runs a column's walk is split
 * into by the sequential kernels (process-wide; for tests and
 * measurements); <= 0 removes the bound (the default: the library's
 * choice by shape and device).  With one run per column nothing is
 * exchanged between CTAs.
 */
wkv_status wkv_debug_set_max_runs(int runs);

/*
 * wkv_debug_set_chain_len: > 0 makes the sequential forward pass walk each
 * column as a chain of runs of that many chunks (each run summarised, then
 * walked again from the state carried in from the run before it, taken
 * from a tagged record); 0 restores the default, which chains runs only
 * when a shape's inputs exceed the L2 cache while its columns leave SMs
 * idle (a long sequence).  Process-wide; for tests and measurements.
 */
wkv_status wkv_debug_set_chain_len(int chunks);

/*
 * wkv_scan_strategy: the strategy wkv_forward and wkv_backward take for a
 * [B, T, C] call on the current device under the current scan mode:
 * WKV_SCAN_CHUNKED or WKV_SCAN_SEQUENTIAL; -1 for invalid sizes or when the
 * device cannot be queried.  Host only; nothing is launched.
 */
int wkv_scan_strategy(int B, int T, int C);

#ifdef __cplusplus
}
#endif

#endif /* WKV_H_ */
