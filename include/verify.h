/*
 * verify.h - C ABI of the exact width-k verification pass (one GB300, sm_103a).
 *
 * A speculative-decoding verify pass runs a block of k draft rows (k = 1..32;
 * the pages measure 1..9) through the target model in one pass and must give,
 * row for row, what k ordinary one-row steps give.  This library provides the
 * data-parallel hot path of that pass for hybrid Gated-DeltaNet / MoE models:
 *
 *   q4_qmv_k            affine 4-bit (group 64) weight x k BF16 rows
 *   q4_gather_experts_k routed top-k experts: fused gate/up + SwiGLU + down +
 *                       fixed-order combine (optionally a sigmoid-gated shared
 *                       expert)
 *   gdn_verify_k        k-row Gated DeltaNet step with per-row state snapshots
 *   gdn_commit          accepted-prefix rollback by slot (pointer) swap
 *   verify_rmsnorm_k    the layer glue norm used by a full verify layer
 *   attn_verify_k       width-k grouped-query attention over an F16 KV cache
 *                       (attn_commit: the cache's rollback)
 *   verify_accept_greedy greedy acceptance of the block on the device, fused
 *                       with the commit of every GDN state (gdn_commit_dev:
 *                       the same commit for any sampler's accepted count)
 *
 * Sources (pages, cited by title and section):
 *   [T]  "Flash-Next optimization transfer to Ornith and Qwen 27B":
 *        table "Shared architecture and implemented paths" and section
 *        "Exact verification kernels and benchmark admission".
 *   [R]  "Red Lite dev45 - speculative decoding with the Qwen3-Next MTP block":
 *        sections "What it is" (2-row verify), "Acceptance" and "Tried and
 *        kept or not".
 *   [F]  "QWEN38FLASH.md - Plan for supporting Qwen/Qwen3.8-Flash-Next":
 *        section 2.1 "Gated DeltaNet (GDN)", 2.3 "MoE", 2.4 (norm forms),
 *        3.1 (KDA -> GDN adaptations), 5.1 (GDN kernel list).
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Memory: every tensor argument is a DEVICE pointer owned by the caller
 *    (cudaMalloc / PyTorch).  The library never frees or keeps caller memory
 *    beyond the call.  verify_init allocates the library's own scratch on the
 *    chosen device; verify_destroy frees it.  Host pointers are rejected with
 *    VERIFY_EINVAL (checked with cudaPointerGetAttributes).
 *  - Streams: every compute call is asynchronous on the caller's stream
 *    (a cudaStream_t passed as `struct CUstream_st*`; NULL = legacy default
 *    stream).  Nothing synchronises the host.  Calls that share one ctx
 *    share its scratch, so they must be ordered on one stream (or otherwise
 *    serialised); concurrent calls on one ctx from different streams race.
 *  - Errors: each call returns a verify_status.  Argument errors are found on
 *    the host before anything is launched (the call then has no effect).
 *    VERIFY_ECUDA reports a launch error.  Kernels never trap: a device-side
 *    problem (a pipeline wait that timed out, an out-of-range expert index)
 *    sets the ctx's device error word, read by verify_device_status.
 *    verify_last_error returns a static, human-readable string for the last
 *    failing call on that ctx.
 *  - BF16 tensors are passed as uint16_t bit patterns.  Outputs requested as
 *    VERIFY_BF16 are the round-to-nearest-even of the fp32 result.
 *  - Exactness (the property the pages require, [T] "Exact verification
 *    kernels", [R] "What it is": "each row in exactly the 1-row kernel's
 *    order"): for every call, row r of a width-k result is bit-identical to a
 *    width-1 call on row r alone.  Accumulation is fp32 in an order that
 *    depends only on the matrix shape and the GPU, never on k or on the other
 *    rows.
 */
#ifndef VERIFY_H_
#define VERIFY_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* == cudaStream_t without pulling in CUDA headers */

typedef enum {
  VERIFY_OK = 0,
  VERIFY_EINVAL = 1,       /* null / host / misaligned pointer, bad size, bad state */
  VERIFY_EUNSUPPORTED = 2, /* k out of range, K % 64 != 0, group != 64, bits != 4,
                              shapes above the library's limits */
  VERIFY_ECUDA = 3,        /* a CUDA runtime call or kernel launch failed */
  VERIFY_EDEVICE = 4       /* a kernel reported an error in the device error word */
} verify_status;

typedef enum {
  VERIFY_F32 = 0,     /* write fp32 */
  VERIFY_BF16 = 1,    /* write bf16 (RNE of the fp32 result) */
  VERIFY_F32_ADD = 2  /* y(fp32) += result: the residual add of a verify layer */
} verify_dtype;

#define VERIFY_MAX_K 32          /* widest verify block any call accepts */
#define VERIFY_PASS_K 16         /* rows per pass: wider blocks run as two passes */
#define VERIFY_GDN_MAX_SLOTS 33  /* VERIFY_MAX_K + 1 state slots */

typedef struct verify_ctx verify_ctx;

/*
 * One affine Q4 matrix with group size 64 ([T] table "Shared architecture":
 * "affine Q4, group size 64, and compatible BF16 tensors"):
 *   weight : w[n][c] = scale[n][c/64] * q[n][c] + bias[n][c/64],  q in 0..15
 * in one of two layouts (`layout`):
 *
 * VERIFY_Q4_ROWS - the affine convention of the MLX runtime [T] uses; the
 * form weights arrive in, accepted only by q4_tile:
 *   packed : uint32 [n_out, k_in/8], row-major; input column c of row n is
 *            bits 4*(c%8) .. 4*(c%8)+3 of packed[n*(k_in/8) + c/8]
 *            (lowest nibble = lowest column).
 *   scales : bf16 [n_out, k_in/64];  biases : bf16 [n_out, k_in/64]
 *   Requirements: packed 16-byte aligned; scales, biases 2-byte aligned.
 *
 * VERIFY_Q4_TILED / VERIFY_Q4_TILED_GATE_UP / VERIFY_Q4_TILED_DOWN - the
 * library's layouts, written by q4_tile, taken by the compute calls:
 * `packed` points to the tiled bytes (16-byte aligned), scales and biases
 * are NULL (they live inside the tiles).  Each (128-row tile, column chunk)
 * is one contiguous block: the tile's scales and biases, then its codes in
 * the order the kernels consume them, so that a pipeline stage is one bulk
 * copy and HBM is read in long runs.
 *   TILED         - dense products (q4_qmv_k, the LM head): 256-column
 *                   chunks.
 *   TILED_GATE_UP - routed and shared experts' fused gate/up matrix
 *                   [2I, n_in], whose tiles pair 64 gate rows with the 64 up
 *                   rows of the same outputs; 128-column chunks.
 *   TILED_DOWN    - routed and shared experts' down matrix; 128-column
 *                   chunks.
 * The experts' smaller blocks let their kernel keep a deeper pipeline in
 * the same shared memory.
 *
 * Requirements: k_in % 64 == 0, k_in >= 64; group_size == 64; bits == 4.
 */
typedef enum {
  VERIFY_Q4_ROWS = 0,
  VERIFY_Q4_TILED = 1,
  VERIFY_Q4_TILED_GATE_UP = 2,
  VERIFY_Q4_TILED_DOWN = 3
} verify_q4_layout;

/* What a matrix is tiled for (q4_tile, q4_tiled_bytes). */
typedef enum {
  VERIFY_TILE_DENSE = 0,   /* -> VERIFY_Q4_TILED */
  VERIFY_TILE_GATE_UP = 1, /* -> VERIFY_Q4_TILED_GATE_UP (n_out = 2I, I % 64 == 0) */
  VERIFY_TILE_DOWN = 2     /* -> VERIFY_Q4_TILED_DOWN */
} verify_tile_kind;

typedef struct {
  const uint32_t* packed;
  const uint16_t* scales;
  const uint16_t* biases;
  int32_t n_out;
  int32_t k_in;
  int32_t group_size; /* must be 64 */
  int32_t bits;       /* must be 4 */
  int32_t layout;     /* verify_q4_layout */
} verify_q4_weight;

/*
 * A stack of n_experts matrices of identical shape, stored back to back
 * (row layout: packed [E, n_out, k_in/8], scales/biases [E, n_out, k_in/64];
 * tiled layout: E tiled matrices).  `w` holds the per-expert shape and the
 * pointers to expert 0.
 */
typedef struct {
  verify_q4_weight w;
  int32_t n_experts;
} verify_q4_experts;

/* ---------------------------------------------------------------- context */

/* Creates a context on `device` (makes it current) and allocates the
 * library's scratch there.  *out receives the context.  The scratch is sized
 * for the limits listed with each call. */
verify_status verify_init(int device, verify_ctx** out);

/* Frees the scratch and the context.  Synchronises the device first. */
verify_status verify_destroy(verify_ctx* ctx);

/* Static string describing the last failing call on ctx ("" if none). */
const char* verify_last_error(const verify_ctx* ctx);

/* Synchronises `stream`, reads and clears the device error word.  Returns
 * VERIFY_OK if no kernel reported a problem since the last check, else
 * VERIFY_EDEVICE with *code (if non-NULL) set to the first error code:
 * 1 = pipeline wait timed out, 2 = expert index out of range, 3 = a device
 * commit found no matching verify pending (nothing committed), 4 = a
 * device-held committed slot outside 0 .. n_slots-1 (the verify wrote nothing). */
verify_status verify_device_status(verify_ctx* ctx, struct CUstream_st* stream, int32_t* code);

/* Number of kernels the library launched on this ctx since verify_init. */
int64_t verify_launch_count(const verify_ctx* ctx);

/* Test aid for failure detection: launches one kernel on `stream` whose two
 * bounded waits are made to run out - a pipeline barrier that nothing arrives
 * on and a counter that nothing increments - through the same wait code and
 * limit (about 2 s at full clock) as the verify kernels.  The kernel then
 * returns; it neither hangs nor faults.  Afterwards verify_device_status
 * reports VERIFY_EDEVICE with code 1 (and clears it), and the context stays
 * usable.  One kernel launch. */
verify_status verify_selftest_stuck_wait(verify_ctx* ctx, struct CUstream_st* stream);

/* ------------------------------------------------------------- q4_tile */

/*
 * Bytes of the tiled layout (kind: verify_tile_kind) of n_experts matrices
 * [n_out, k_in]; -1 for invalid shapes or kind.  Equals the row layout's
 * bytes when n_out % 128 == 0, plus the zero rows that complete the last
 * 128-row tile otherwise.
 */
int64_t q4_tiled_bytes(int32_t n_out, int32_t k_in, int32_t n_experts, int32_t kind);

/*
 * Converts src (VERIFY_Q4_ROWS; n_experts matrices back to back) into the
 * tiled layout of `kind` (verify_tile_kind) at dst (device, 16-byte aligned,
 * dst_bytes >= q4_tiled_bytes) on `stream`, and fills *out (a host struct)
 * with the tiled description: packed = dst, layout = VERIFY_Q4_TILED,
 * VERIFY_Q4_TILED_GATE_UP or VERIFY_Q4_TILED_DOWN.  A one-time step when
 * weights are loaded; src may be freed once the stream has passed the
 * conversion.  Every bit of src is kept: the tiled matrix computes exactly
 * what src describes.  Returns VERIFY_EUNSUPPORTED for an unknown kind.
 */
verify_status q4_tile(verify_ctx* ctx, const verify_q4_weight* src, int32_t n_experts, int32_t kind, void* dst,
                      int64_t dst_bytes, verify_q4_weight* out, struct CUstream_st* stream);

/* ------------------------------------------------------------ q4_qmv_k */

/*
 * Dense width-k product ([T] "Exact verification kernels": the small-batch
 * Q4 kernel at widths 4/8/9 agrees exactly with serial QMV; [R] "What it is":
 * two-vector kernels decode each weight once and compute each row in the
 * 1-row kernel's order):
 *
 *     y[r][n] = sum_c w[n][c] * x[r][c]      r < k, n < n_out
 *
 * W : VERIFY_Q4_TILED.
 * x : bf16 [k, k_in] row-major, 16-byte aligned.
 * y : [k, n_out] row-major, fp32 (VERIFY_F32 / VERIFY_F32_ADD) or bf16.
 * k : 1..VERIFY_MAX_K.   Limits: n_out <= 1<<20, k_in <= 1<<17.
 * Each packed weight is read from HBM once per pass of up to VERIFY_PASS_K
 * rows: k <= 16 is one launch, 17..32 two launches (rows 0..15, then the
 * rest), each row computed as in a width-1 call.
 */
verify_status q4_qmv_k(verify_ctx* ctx, const verify_q4_weight* W,
                       const uint16_t* x, int k, void* y, int dtype_out,
                       struct CUstream_st* stream);

/* ------------------------------------------------- q4_gather_experts_k */

/*
 * Routed mixture-of-experts for k rows ([T] "Exact verification kernels":
 * gathered expert kernel, affine Q4/group-64, top-8 of 256, fused gate/up;
 * [R] "What it is": all rows' (expert,row) pairs in one dispatch and one
 * tail; [F] 2.3: gate+up concatenated [E, 2I, H], SwiGLU, a sigmoid-gated
 * shared expert).  Per row r:
 *
 *   idx[r][0..T)  = the T largest router logits of row r, in descending
 *                   order (equal logits: lower expert index first)
 *   wts[r][j]     = exp(l_j - l_0) / sum_{j'<T} exp(l_j' - l_0)
 *                   (softmax over all E, keep T, renormalise == softmax of
 *                   the T selected logits)
 *   for j < T, e = idx[r][j]:
 *     g = W_gu[e][0..I)  . x[r],  u = W_gu[e][I..2I) . x[r]
 *     h = bf16( silu(g) * u )                          (silu(t) = t/(1+e^-t))
 *     p_j = W_d[e] . h
 *   y[r] = sum_{j=0..T-1} wts[r][j] * p_j    (ascending j, fp32)
 *   if a shared expert is given: y[r] += sigmoid(sg[r]) * (W_sd . bf16(silu(W_sgu[0..I).x) * W_sgu[I..2I).x))
 *
 * gate_up : experts [E, 2I, H], VERIFY_Q4_TILED_GATE_UP;
 * down    : experts [E, H, I], VERIFY_Q4_TILED_DOWN.
 * logits  : fp32, row r at logits + r*logits_ld, E entries.
 * x       : bf16 [k, H].   idx_out : int32 [k, T];  w_out : fp32 [k, T].
 * y       : fp32 [k, H] (VERIFY_F32 or VERIFY_F32_ADD) or bf16.
 * shared_gate_up [2I, H] (TILED_GATE_UP), shared_down [H, I] (TILED_DOWN), shared_gate_logit (fp32, row r
 * at shared_gate_logit + r*logits_ld) may all be NULL (no shared expert).
 * Limits: E <= 512, 1 <= T <= 16, 64 <= H <= 8192, 64 <= I <= 4096,
 * H % 64 == I % 64 == 0.
 * Expert weights are read once per pass of up to VERIFY_PASS_K rows for
 * every distinct expert the pass selects (the union of its rows' routes).
 * Two kernel launches per pass on `stream`: the routed experts (gate/up and
 * down items in one kernel), then the combine; k in 17..32 runs two passes
 * (rows 0..15, then the rest).
 */
verify_status q4_gather_experts_k(verify_ctx* ctx,
                                  const verify_q4_experts* gate_up,
                                  const verify_q4_experts* down,
                                  const float* logits, int64_t logits_ld,
                                  int top_k, const uint16_t* x, int k,
                                  int32_t* idx_out, float* w_out,
                                  void* y, int dtype_out,
                                  const verify_q4_weight* shared_gate_up,
                                  const verify_q4_weight* shared_down,
                                  const float* shared_gate_logit,
                                  struct CUstream_st* stream);

/* ------------------------------------------------------- gdn_verify_k */

/*
 * Gated DeltaNet layer geometry and parameters ([F] 2.1, 3.1):
 *   C = 2*n_qk_heads*head_dim_k + n_v_heads*head_dim_v conv channels
 *   (q | k | v, in that order).  V head h uses QK head h / (n_v_heads/n_qk_heads).
 * conv_w  : fp32 [C, conv_kernel]; tap conv_kernel-1 multiplies the current row.
 * A_log, dt_bias : fp32 [n_v_heads].   norm_w : fp32 [head_dim_v].
 * Supported: head_dim_k == head_dim_v in {32, 64, 128}, conv_kernel == 4,
 * n_v_heads % n_qk_heads == 0.
 */
typedef struct {
  int32_t n_qk_heads, n_v_heads, head_dim_k, head_dim_v, conv_kernel;
  float q_scale;  /* multiplies the L2-normalised q (1/sqrt(head_dim_k)) */
  float l2_eps;   /* q,k L2 norm: x / sqrt(sum x^2 + l2_eps) (1e-6) */
  float norm_eps; /* gated RMSNorm epsilon (1e-6) */
  int32_t gate_act; /* 0 = sigmoid (default), 1 = silu */
  const float* conv_w;
  const float* A_log;
  const float* dt_bias;
  const float* norm_w;
} verify_gdn_params;

/*
 * Recurrent state of one GDN layer as a ring of caller-allocated slots.
 * Slot s holds S_slots[s]: fp32 [n_v_heads, head_dim_v, head_dim_k]
 * (S[h][i][j], i = value row, j = key column) and conv_slots[s]: bf16
 * [conv_kernel-1, C] (the last conv_kernel-1 input rows, oldest first).
 * `cur` is the committed slot.  After gdn_verify_k(k), pending[r] is the slot
 * that holds the state after the first r rows (pending[0] == cur) and
 * pending_k == k; gdn_commit turns one of them into `cur`.
 * The caller fills S_slots/conv_slots/n_slots/cur once (n_slots >= k+1 for
 * every verify) and then only reads the struct.
 *
 * Device-held commit (dev != NULL, set by gdn_state_to_device): the committed
 * slot lives in device memory, dev[0] = committed slot, dev[1] = rows of the
 * verify still pending (0: none), so that an accept and commit on the device
 * (verify_accept_greedy, gdn_commit_dev) need no host round trip and a
 * captured CUDA graph of verify + accept stays valid from step to step.  The
 * kernels then read and advance dev; the host fields cur, pending_k and
 * pending are not used, and the host commits reject the state.  Slots are used
 * in the same order as with a host-held commit: the state after the first r
 * rows goes to slot r-1 + (r-1 >= cur), the r-th slot other than cur.
 */
typedef struct {
  float* S_slots[VERIFY_GDN_MAX_SLOTS];
  uint16_t* conv_slots[VERIFY_GDN_MAX_SLOTS];
  int32_t n_slots;
  int32_t cur;
  int32_t pending_k;
  int32_t pending[VERIFY_GDN_MAX_SLOTS];
  int32_t* dev; /* NULL, or device int32 [2] as above */
} verify_gdn_state;

/* Inputs of a width-k GDN call: bf16, row r of each at ptr + r*ld.  qkv has
 * C entries per row, z n_v_heads*head_dim_v, a and b n_v_heads each. */
typedef struct {
  const uint16_t* qkv; int64_t ld_qkv;
  const uint16_t* z;   int64_t ld_z;
  const uint16_t* a;   int64_t ld_a;
  const uint16_t* b;   int64_t ld_b;
} verify_gdn_inputs;

/*
 * k-row Gated DeltaNet step ([F] 2.1 per-token pipeline and delta rule;
 * [R] "What it is": row r runs from row r-1's state and the state after
 * each row is written to snapshot buffers inside the kernels; [T] table
 * "Fused GDN preparation" widths 1..9).  Starting from slot st->cur, for
 * r = 0..k-1 and every V head h (QK head hq):
 *   conv:   c = silu(sum_t conv_w[ch][t] * window_r[t]) per channel, window_r
 *           = the conv_kernel most recent input rows ending at row r
 *   q = c[q channels of hq] / sqrt(|.|^2 + l2_eps) * q_scale
 *   kk = c[k channels of hq] / sqrt(|.|^2 + l2_eps);  v = c[v channels of h]
 *   beta = sigmoid(b[r][h]);  g = exp(-exp(A_log[h]) * softplus(a[r][h] + dt_bias[h]))
 *   S <- g*S;  m = S.kk;  delta = (v - m)*beta;  S[i][j] += delta[i]*kk[j];  y = S.q
 *   o[r][h*dv + i] = y_i / sqrt(mean(y^2) + norm_eps) * norm_w[i] * act(z[r][h*dv+i])
 * The state (S and conv window) after row r is written to slot pending[r+1]
 * (the free slots in ascending index order); slot cur is only read.
 * o : [k, n_v_heads*head_dim_v] fp32 or bf16 (VERIFY_F32 / VERIFY_BF16).
 * Requires n_slots >= k+1, all slot pointers 16-byte aligned.  One launch for
 * k <= 16; k in 17..32 adds a second launch that continues from the snapshot
 * after row 15 (the state carries over exactly).
 * A second verify without a commit in between starts again from `cur`.
 * With a device-held commit (st->dev) the kernel takes cur from dev[0] when
 * it runs, every one of the n_slots slots must be valid, and dev[1] becomes k.
 */
verify_status gdn_verify_k(verify_ctx* ctx, const verify_gdn_params* p,
                           verify_gdn_state* st, const verify_gdn_inputs* in,
                           int k, void* o, int dtype_out,
                           struct CUstream_st* stream);

/*
 * Accepted-prefix rollback ([R] "What it is": a rejected draft is undone by
 * swapping the DeltaNet state pointers with the snapshots; "Acceptance").
 * Makes the state after the first `accepted` rows of the last verify current:
 * cur = pending[accepted]; accepted = 0 keeps the pre-verify state.
 * Host-only, O(1), touches no device memory and launches nothing.
 * Errors: VERIFY_EINVAL if nothing is pending (a second commit), accepted
 * is outside 0..pending_k, or the state's commit is device-held.
 */
verify_status gdn_commit(verify_gdn_state* st, int accepted);

/* gdn_commit(&states[l], accepted) for l = 0 .. n_states - 1, all or nothing:
 * every state is checked first (VERIFY_EINVAL, nothing changed, if any would
 * be rejected).  Host-only. */
verify_status gdn_commit_all(verify_gdn_state* states, int n_states, int accepted);

/* ------------------------------------------ acceptance and commit on device */

/*
 * Moves the committed slot of states[0 .. n_states-1] to the device: dev is
 * caller-owned device memory of int32 [n_states][2]; states[l].dev becomes
 * dev + 2*l, holding {states[l].cur, 0}.  A verify still pending on the host
 * is dropped (as a second verify would drop it).  Copies on `stream` and
 * synchronises it.  VERIFY_EINVAL: NULL or misaligned dev, a state already on
 * the device, a cur outside 0 .. n_slots-1.
 */
verify_status gdn_state_to_device(verify_ctx* ctx, verify_gdn_state* states, int n_states, int32_t* dev,
                                  struct CUstream_st* stream);

/*
 * Back to a host-held commit: synchronises `stream`, copies each dev[0] into
 * cur, sets pending_k = 0 (a verify pending on the device is dropped) and
 * dev = NULL.  VERIFY_EINVAL if a state is not on the device or holds an
 * invalid slot (then nothing changes).
 */
verify_status gdn_state_to_host(verify_ctx* ctx, verify_gdn_state* states, int n_states,
                                struct CUstream_st* stream);

/*
 * Rollback by slot swap on the device ([R] "What it is": a rejected draft is
 * undone by swapping the DeltaNet state pointers with the snapshots), with the
 * accepted row count read from device memory (*accepted, any sampler's):
 * for every state, all or nothing, cur <- accepted == 0 ? cur
 * : accepted-1 + (accepted-1 >= cur), and nothing is pending afterwards.  The
 * states must have consecutive dev words (states[l].dev == states[0].dev + 2l,
 * as gdn_state_to_device sets them).  Errors found on the host return
 * VERIFY_EINVAL before the launch; on the device, a state with no verify
 * pending or accepted outside 0 .. pending rows commits nothing and records
 * device error 3.  One kernel launch.
 */
verify_status gdn_commit_dev(verify_ctx* ctx, const verify_gdn_state* states, int n_states,
                             const int32_t* accepted, struct CUstream_st* stream);

/*
 * Greedy acceptance of a width-k verify block, fused with the commit
 * ([R] "What it is": the pending token and the drafts run as the rows of one
 * pass; "Acceptance": a draft stands when the token chosen from the previous
 * row's logits equals it, so greedy verification gives serial decoding's
 * tokens exactly).  Inputs:
 *   logits : device fp32 [k, V], row r at logits + r*ld: the target's logits
 *            after row r (row 0 the pending token, row r >= 1 draft d_r);
 *   draft  : device int32 [k-1], draft[r-1] = d_r (may be NULL when k == 1).
 * Computes t_r = argmax_v logits[r][v] (lowest index among equal maxima,
 * -0 == +0, a NaN above every number: numpy's argmax), m = the number of
 * leading drafts with d_{r+1} == t_r, and writes
 *   result : device int32 [2 + k] = { a = m + 1, t_m, t_0, ..., t_{k-1} }
 * (a rows stand; t_m is the next pending token).  If n_states > 0 it then
 * commits a on every state as gdn_commit_dev does, which also requires each
 * state's pending rows to equal k (else device error 3, nothing committed).
 * Limits: 1 <= k <= 32, 1 <= V <= 2^30, ld >= V.  Rows that are 16-byte
 * aligned (logits aligned, ld % 4 == 0) are read as float4.  One kernel
 * launch; the ctx's scratch serialises calls on one ctx (one stream at a time).
 */
verify_status verify_accept_greedy(verify_ctx* ctx, const float* logits, int64_t ld, int V, int k,
                                   const int32_t* draft, int32_t* result, const verify_gdn_state* states,
                                   int n_states, struct CUstream_st* stream);

/*
 * GPU token selection at the target, fused ([T] table "Shared architecture":
 * greedy proposals use a compact vocabulary, target verification the full
 * one; [R] "Acceptance"): the LM head product y = W . x[r] (as q4_qmv_k
 * computes it) with an argmax epilogue, so the logits never reach memory,
 * then greedy acceptance and the commit as verify_accept_greedy does.
 *   W     : VERIFY_Q4_TILED [V, H], V = vocabulary (n_out <= 2^20).
 *   x     : bf16 [k, H] (the final-normed rows), 16-byte aligned.
 *   draft, result, states, n_states: as verify_accept_greedy.
 * The choices equal those of q4_qmv_k followed by verify_accept_greedy on its
 * fp32 output, bit for bit.  One launch per pass of up to 16 rows (17..32 rows:
 * two passes), whose epilogue merges each row's argmax key with a 64-bit
 * atomicMax, then a one-CTA launch for the accepted prefix and the commit.
 * Shares the acceptance scratch of the ctx with verify_accept_greedy.
 */
verify_status verify_lm_head_accept(verify_ctx* ctx, const verify_q4_weight* W, const uint16_t* x, int k,
                                    const int32_t* draft, int32_t* result, const verify_gdn_state* states,
                                    int n_states, struct CUstream_st* stream);

/* ---------------------------------------------------- attention verify */

/*
 * Grouped-query attention of a verify layer ([F] 2.2: 24 query and 2 KV
 * heads of dim 256, RoPE on the first 64 dims with base 1e7, a sigmoid gate on
 * the output, an F16 KV cache; below its 2048-token sparse budget QSA is this
 * dense attention).
 */
typedef struct {
  int32_t n_q_heads, n_kv_heads; /* n_q_heads a multiple of n_kv_heads */
  int32_t head_dim;              /* 128 or 256 */
  int32_t rope_dim;              /* even, <= head_dim: the rotated leading dims */
  float rope_theta;
} verify_attn_params;

/*
 * KV cache of one attention layer, caller-allocated: K and V are binary16
 * [n_kv_heads, capacity, head_dim]; positions 0 .. len-1 are committed.
 * split (a multiple of 32, >= 32) fixes how the key positions are cut for
 * the split-KV kernel: [s*split, (s+1)*split).  Results are bit-identical
 * across widths (row r of a width-k call == a width-1 call at len + r) for
 * one split value.  K and V must be 16-byte aligned device memory (the
 * split kernel reads them with TMA tile loads).  work: caller device memory
 * of attn_workspace_bytes(...) bytes, 256-byte aligned (the rotated queries
 * and the partial results).  After attn_verify_k(k)
 * the block's keys and values sit at len .. len+k-1 and pending_k == k;
 * attn_commit(a) makes a of them committed (len += a); the others are
 * overwritten by the next verify.
 */
typedef struct {
  uint16_t* K;
  uint16_t* V;
  int64_t capacity;
  int32_t len;
  int32_t split;
  int32_t pending_k;
  void* work;
  int64_t work_bytes;
} verify_kv_cache;

/* Inputs of a width-k attention call, bf16, row r at ptr + r*ld: q and gate
 * [n_q_heads*head_dim] (head-major), k and v [n_kv_heads*head_dim]. */
typedef struct {
  const uint16_t* q;    int64_t ld_q;
  const uint16_t* gate; int64_t ld_gate;
  const uint16_t* k;    int64_t ld_k;
  const uint16_t* v;    int64_t ld_v;
} verify_attn_inputs;

/* A split for a cache of `capacity` positions: about 74 key splits per KV
 * head at full length (with two KV heads, one wave of one CTA per SM), a
 * multiple of 64 and at least 128. */
int32_t attn_default_split(int64_t capacity);

/* Workspace bytes attn_verify_k needs for a cache of `capacity` positions cut
 * by `split`, for widths up to max_k (0 for bad arguments). */
int64_t attn_workspace_bytes(const verify_attn_params* p, int64_t capacity, int32_t split, int32_t max_k);

/*
 * Width-k attention verify ([R] "What it is": attention runs per row, row r
 * seeing the earlier rows' K/V; [T] "Exact verification kernels": each row's
 * serial KV window).  Row r is the token at position P + r, P = cache->len:
 *   key_r = rope(k[r], P + r) and v[r], rounded to binary16, are written to
 *   the cache at position P + r (every KV head);
 *   for query head h (KV head h / (n_q_heads / n_kv_heads)):
 *     s_j = rope(q[r][h], P + r) . K[j] / sqrt(head_dim),  j = 0 .. P + r
 *     o[r][h*head_dim + i] = (sum_j softmax(s)_j V[j][i]) * sigmoid(gate[r][h*head_dim + i])
 * rope(x, pos) rotates the pair (x_i, x_{i+rope_dim/2}) by the angle
 * pos * theta^(-2i/rope_dim) for i < rope_dim/2; other dims pass through.
 * o: [k, n_q_heads*head_dim], VERIFY_F32 or VERIFY_BF16 (row stride
 * n_q_heads*head_dim).  Three kernel launches (append; split partials on
 * the tcgen05 tensor cores with TMEM accumulators; combine).  Limits: 1 <= k <= 32, k * n_q_heads / n_kv_heads <= 512,
 * len + k <= capacity.  Arithmetic: rotation angles in float64, the
 * rotation in fp32; q.K and p.V on the tensor cores with binary16 operands and
 * fp32 sums, the scaled query and the probabilities each carried as a pair of
 * binary16 values (hi + lo), so that the cache's binary16 values are the only
 * rounding of note.
 */
verify_status attn_verify_k(verify_ctx* ctx, const verify_attn_params* p, verify_kv_cache* cache,
                            const verify_attn_inputs* in, int k, void* o, int dtype_out,
                            struct CUstream_st* stream);

/* Rollback of the cache: len += accepted (0 .. pending_k), nothing pending
 * afterwards.  Host-only.  VERIFY_EINVAL if nothing is pending or accepted is
 * out of range. */
verify_status attn_commit(verify_kv_cache* cache, int accepted);

/* --------------------------------------------------------- layer glue */

/*
 * Row RMSNorm used around a verify layer ([F] 2.4: non-gated norms are
 * zero-centred, y*(1+w)):
 *   out[r][c] = x[r][c] / sqrt(mean_c x[r][c]^2 + eps) * (zero_centered ? 1 + w[c] : w[c])
 * x fp32 [k, n]; w fp32 [n]; out [k, n] bf16 or fp32.  n <= 16384, n % 4 == 0.
 */
verify_status verify_rmsnorm_k(verify_ctx* ctx, const float* x, const float* w,
                               float eps, int zero_centered, int n, int k,
                               void* out, int dtype_out,
                               struct CUstream_st* stream);


/* --------------------------------------------------------- a verify layer */

/*
 * One hybrid verify layer ([F] section 2: every layer is a Gated DeltaNet
 * mixer followed by a MoE FFN; 2.3: 10 routed + 1 shared expert; 2.4:
 * zero-centred norms), applied to the k-row residual stream h (fp32 [k, H],
 * updated in place):
 *   xn  = bf16(rmsnorm_zc(h, norm1_w))
 *   p   = bf16(in_proj . xn)          rows: q|k|v (C), z (Hv*dv), a (Hv), b (Hv)
 *   o   = gdn_verify_k(p...)           bf16; state slots advance as in gdn_verify_k
 *   h  += out_proj . o
 *   xn2 = bf16(rmsnorm_zc(h, norm2_w))
 *   l   = router . xn2                 fp32 [k, E+1]: E routing logits, then the
 *                                      shared expert's gate logit
 *   h  += q4_gather_experts_k(gate_up, down, l[:, :E], top_k, xn2,
 *                             shared_gate_up, shared_down, l[:, E])
 * idx_out (optional, device int32 [k, top_k]) receives the routed expert
 * indices.  Eight kernel launches on `stream` for k <= 16 (fourteen for
 * 17..32: the products, the DeltaNet step and the experts run two passes),
 * no host synchronisation.  Scratch
 * activations live in the context (limits: k <= 32, H <= 8192, in_proj rows
 * <= 32768, E + 1 <= 1024).  Weight shapes must match: in_proj [C + Hv*dv +
 * 2*Hv, H], out_proj [H, Hv*dv], router [E + 1, H], gate_up [E, 2I, H],
 * down [E, H, I], shared_gate_up [2I, H], shared_down [H, I]; all tiled
 * (gate_up and shared_gate_up as VERIFY_Q4_TILED_GATE_UP, down and
 * shared_down as VERIFY_Q4_TILED_DOWN, the rest VERIFY_Q4_TILED).
 */
typedef struct {
  verify_q4_weight in_proj;
  verify_q4_weight out_proj;
  verify_q4_weight router;
  verify_q4_experts gate_up;
  verify_q4_experts down;
  verify_q4_weight shared_gate_up;
  verify_q4_weight shared_down;
  verify_gdn_params gdn;
  const float* norm1_w; /* [H], used as 1 + w */
  const float* norm2_w; /* [H], used as 1 + w */
  float norm_eps;
  int32_t top_k;
} verify_layer;

verify_status verify_layer_k(verify_ctx* ctx, const verify_layer* L, verify_gdn_state* st, float* h, int k,
                             int32_t* idx_out, struct CUstream_st* stream);

/*
 * A verify pass of k rows through n_layers layers in one call: verify_layer_k
 * on (layers[l], states[l]) for l = 0 .. n_layers - 1, in order, on `stream`,
 * h updated in place.  idx_out (optional, device int32) receives layer l's
 * routed indices at idx_out + l * k * layers[l].top_k.  Returns the first
 * failing layer's status; the layers before it have been enqueued and their
 * states advanced.  verify_layer_k's launches per layer, no host
 * synchronisation.  Layer 0's first kernel waits for everything enqueued
 * before the call; each later layer's first kernel is a programmatic
 * dependent of the layer before (it reads only its weights before its
 * dependency wait).
 */
verify_status verify_stack_k(verify_ctx* ctx, const verify_layer* layers, verify_gdn_state* states, int n_layers,
                             float* h, int k, int32_t* idx_out, struct CUstream_st* stream);

/*
 * Profiling aid (no counterpart on the pages): while set, every
 * verify_layer_k call records events[0..7] (cudaEvent_t handles created by the
 * caller with timing enabled) on its stream - before the first norm, then
 * after the norm, in_proj, GDN, out_proj, second norm, router and experts -
 * so the caller can time each sub-step, also inside a captured CUDA graph.
 * A NULL entry skips that point; events = NULL (or n = 0) switches it off.
 * n must be 8.
 */
verify_status verify_set_layer_events(verify_ctx* ctx, void* const* events, int n);

/* ------------------------------------- routed experts without allocation */

/*
 * Routed-expert call that allocates no device memory.  The pages have no
 * counterpart of this entry point; it exists for callers that are not
 * allowed to allocate: for example a host framework that hands out all
 * device memory from its own arena and forbids plug-ins to call cudaMalloc,
 * or a latency-critical serving loop where cudaMalloc/cudaFree would
 * synchronise the device.  Such callers cannot create a verify_ctx (its
 * scratch is allocated), so this call needs none.
 *
 * It computes exactly what q4_gather_experts_k computes, with the same
 * arguments (no ctx) and the same shape rules and status codes, plus
 * `device_error`: an optional device int32 the caller owns, set to 1 if a
 * pipeline wait timed out.  With `device_error` NULL a timeout is not
 * reported anywhere, and idx_out, w_out and y are then undefined: callers
 * that must know pass a word (and zero it before the call).  The
 * caller passes all inputs and outputs; the kernels' scratch (SwiGLU rows,
 * per-rank partial outputs, an error word, the expert kernel's item counter
 * and per-unit counts) lives in one array of
 * VERIFY_NOALLOC_SCRATCH_BYTES compiled into the library, which every GPU
 * that loads the library holds until the process exits.
 *   - Limit: k <= VERIFY_PASS_K (one pass); k*(T+s)*I*2 + k*(T+s)*H*4 bytes (s = 1 with a shared expert, each
 *     part rounded up to 256) plus 5376 must fit the array; larger calls
 *     return VERIFY_EUNSUPPORTED before anything is enqueued.
 *   - The first call on each device sets that device up (resolves the array's
 *     device address, sets the kernels' launch attributes); make that first
 *     call before any stream capture.
 *   - Every call on a device shares the array, which keeps the last call's
 *     contents; the call clears what must start at zero (the error word and
 *     the counters) on `stream` before its kernels.  Calls whose work
 *     overlaps on the GPU (different streams, no ordering) race on it.
 * The calling thread's current device is used.
 */
#define VERIFY_NOALLOC_SCRATCH_BYTES (8u << 20)

verify_status q4_gather_experts_k_noalloc(const verify_q4_experts* gate_up, const verify_q4_experts* down,
                                          const float* logits, int64_t logits_ld, int top_k,
                                          const uint16_t* x, int k, int32_t* idx_out, float* w_out,
                                          void* y, int dtype_out,
                                          const verify_q4_weight* shared_gate_up,
                                          const verify_q4_weight* shared_down,
                                          const float* shared_gate_logit, int32_t* device_error,
                                          struct CUstream_st* stream);

#ifdef __cplusplus
}
#endif

#endif /* VERIFY_H_ */
