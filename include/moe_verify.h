/*
 * moe_verify.h -- C ABI of the GB300 (sm_103a) MoE verify-layer library.
 *
 * The layer is the target model's MoE block inside DFlash target-verified
 * block speculative decoding: K draft rows are verified in one forward; each
 * row is routed top-k over E experts; each selected expert's NVFP4
 * gate/up/down projections and a shared expert are evaluated and combined
 * ("Why this challenge exists", mlxfast Laguna XS 2.1 (DFlash) README:
 * 256 routed experts plus one shared expert, 8 experts per token, MoE
 * intermediate 512, routed/shared projections NVFP4 4-bit group-16, router
 * bf16).  An expert chosen by several rows streams its weights once (PR #844,
 * "8. What I looked at": the routed gather reads an expert once per
 * (row, slot) and has no cross-row dedup).
 *
 * Conventions for every entry point
 *  - All data pointers are DEVICE pointers owned by the caller, 16-byte
 *    aligned.  bf16 tensors are passed as their 16-bit patterns (uint16_t).
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *    asynchronous: they enqueue work and return; nothing blocks the host
 *    except moe_workspace_error().
 *  - The library allocates no memory, reads no environment variables and
 *    keeps no per-call state on the host.  Concurrent calls on different
 *    streams need distinct workspaces.
 *  - Argument errors are detected on the host before anything is enqueued
 *    and returned as a negative moe_status.  A failed launch returns
 *    MOE_ERR_CUDA.  A device-side wait that ran out of time is recorded in
 *    the workspace and read back with moe_workspace_error().
 *  - Results are deterministic: identical inputs give bit-identical outputs
 *    (no floating-point atomics; every reduction has a fixed order).
 */
#ifndef MOE_VERIFY_H
#define MOE_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,        /* null pointer, K/shape out of range */
  MOE_ERR_UNSUPPORTED_SHAPE = -2,  /* shape outside the supported envelope */
  MOE_ERR_WORKSPACE_TOO_SMALL = -3,
  MOE_ERR_MISALIGNED = -4,         /* a pointer is not 16-byte aligned */
  MOE_ERR_CUDA = -5,               /* a CUDA runtime/driver call failed */
  MOE_ERR_DEVICE_TIMEOUT = -6,     /* a bounded device-side wait expired */
  MOE_ERR_CAPACITY = -7            /* a KV cache append past the cache's capacity */
} moe_status;

/*
 * One NVFP4 projection over a stack of experts, [n_exp][rows][cols]
 * (cols is the reduction dimension).  Element (e, r, c) has the value
 *   e2m1(code) * e4m3(scale) * tensor_scale[e]
 * where code is the low nibble of codes[e][r][c/2] for even c and the high
 * nibble for odd c (E2M1: sign, 2 exponent bits with bias 1, 1 mantissa
 * bit), scale = scales[e][r][c/16] (OCP E4M3FN), one scale per 16
 * consecutive columns of a row.
 */
typedef struct {
  const uint8_t* codes;         /* [n_exp][rows][cols/2] */
  const uint8_t* scales;        /* [n_exp][rows][cols/16] */
  const float* tensor_scale;    /* [n_exp] */
} moe_nvfp4;

/*
 * Router scoring (moe_layer.scoring).
 *  MOE_SCORE_SOFTMAX  probabilities softmax(logit + bias) over all experts;
 *                     the top_k largest logit + bias are selected and their
 *                     probabilities renormalised over the selection.
 *  MOE_SCORE_SIGMOID  the router tail of the Laguna checkpoint (PR #844,
 *                     "4. What I ported", router-tail row; "5. Numerical
 *                     safety": renormalised top-k, routed scaling 2.5):
 *                     scores s = sigmoid(logit) in FP32, the bias added to
 *                     the scores for the selection only (the top_k largest
 *                     s + bias), weights = the selected s / their sum.
 *                     The sigmoid is one fixed sequence of correctly rounded
 *                     FP32 operations, so the selection is reproducible:
 *                       l <- clamp(l, -80, 80), t = -l,
 *                       n = rint(t * log2 e), r = t - n ln2 (ln 2 split in a
 *                       16-bit head and a tail, two fused multiply-adds),
 *                       e = (degree-7 Taylor polynomial of e^r) * 2^n,
 *                       s = 1 / (1 + e).
 */
#define MOE_SCORE_SOFTMAX 0
#define MOE_SCORE_SIGMOID 1

/*
 * One MoE layer.  gate/up: rows = inter, cols = hidden; down: rows = hidden,
 * cols = inter; the sh_* projections hold one expert of intermediate
 * shared_inter (0 = no shared expert, the sh_* fields are then ignored).
 * Supported envelope: hidden in {256, 512, ..., 2048} (a multiple of 256);
 * inter in {128, 256, 512}; shared_inter in {0, inter}; 1 <= top_k <= 32;
 * top_k <= n_experts <= 1024.  Outside it: MOE_ERR_UNSUPPORTED_SHAPE.
 */
typedef struct {
  int hidden, n_experts, top_k, inter, shared_inter;
  float routed_scale;          /* multiplies the routed sum (1.0 = none) */
  const uint16_t* router_w;    /* bf16 [n_experts][hidden] */
  const float* router_bias;    /* [n_experts] or NULL = 0: added to the logits
                                  (softmax scoring) or to the sigmoid scores
                                  for the selection only (sigmoid scoring) */
  moe_nvfp4 gate, up, down;
  moe_nvfp4 sh_gate, sh_up, sh_down;
  int scoring;                 /* MOE_SCORE_SOFTMAX (0) or MOE_SCORE_SIGMOID */
} moe_layer;

/* Largest number of verify rows one call accepts. */
#define MOE_MAX_ROWS 16

/*
 * Bytes of device workspace a layer call with K rows needs (0 on an invalid
 * layer or K).  The workspace must be zero-filled once before its first use
 * (e.g. cudaMemsetAsync); every call leaves it ready for the next call,
 * with any K and layer whose size fits in it.  After a call that returned
 * MOE_ERR_DEVICE_TIMEOUT zero-fill it again.
 */
size_t moe_verify_layer_workspace_size(const moe_layer* layer, int K);

/*
 * Router: logits = x_norm . router_w^T + bias in one fixed FP32 order, a
 * softmax over all experts, the top_k experts per row (larger logit first,
 * lower expert index on an exact tie), and their probabilities renormalised
 * over the selected set (PR #844, "4. What I ported": top-k selection and
 * renormalisation of the router scores).
 *   x_norm  bf16 [K][hidden] (already normalised)
 *   idx     int32 [K][top_k] out, rank order;  w  float [K][top_k] out
 *   group   int32 out (nullable): experts grouped for dedup,
 *           with G = min(n_experts, K*top_k):
 *             group[0]                 n = number of distinct experts
 *             group[1 .. 1+G)          the distinct experts ascending, then -1
 *             group[1+G .. 2+2G)       offsets; expert u owns pair slots
 *                                      [off[u], off[u+1]); off[u] = K*top_k for u >= n
 *             group[2+2G .. 2+2G+K*top_k)  pair ids r*top_k + s, rows ascending
 *           (moe_group_ints(K, n_experts, top_k) ints)
 *   ws      workspace of moe_verify_layer_workspace_size(layer, K) bytes
 */
moe_status moe_router_topk(const moe_layer* layer, const uint16_t* x_norm, int K, int32_t* idx,
                           float* w, int32_t* group, void* ws, size_t ws_bytes, void* stream);

/* Number of int32 entries of the group output. */
size_t moe_group_ints(int K, int n_experts, int top_k);

/*
 * The MoE verify layer:
 *   y_r = bf16( routed_scale * sum_{s<top_k} w_{r,s} * Down_e(h_{r,s})
 *               + Down_sh(h_sh) + residual_r ),   e = idx[r][s]
 *   h = bf16( silu(Gate_e x_r) * (Up_e x_r) )
 * (PR #844, "4. What I ported" and "5. Numerical safety": silu(gate)*up,
 * weighted expert sum, routed scaling, shared add and decoder residual add
 * in that order).  Each distinct expert's weights are read once per call.
 * The combine is one FP32 expression per output, each operation rounded
 * (no fused multiply-add), one bf16 rounding at the end:
 *   acc = 0;  acc = acc + w_{r,s} * d_{r,s}  for s = 0 .. top_k-1
 *   y   = bf16( ((routed_scale * acc) + d_sh) + residual )
 *   x_norm    bf16 [K][hidden], the normalised block input
 *   residual  bf16 [K][hidden] or NULL
 *   y         bf16 [K][hidden] out (may alias residual, not x_norm)
 *   idx_out, w_out, group_out: optional copies of the routing (as in
 *             moe_router_topk); NULL to skip
 * Accumulation is FP32; activations enter the tensor cores as FP16 after an
 * exact per-row power-of-two rescaling, so no bf16 value overflows.
 *
 * The call is one grid of one CTA per SM whose CTAs wait on one another
 * (every wait bounded, MOE_ERR_DEVICE_TIMEOUT when it runs out).  It needs
 * all SMs of the GPU within that bound: work that holds SMs briefly
 * (another kernel finishing) only delays it, but two layer calls (this one,
 * moe_verify_stack or moe_verify_step) running at the same time on one GPU,
 * e.g. on two streams, can each hold part of the SMs and both time out.
 * Serialise them (one stream, or events between the streams).
 */
moe_status moe_verify_layer(const moe_layer* layer, const uint16_t* x_norm, int K,
                            const uint16_t* residual, uint16_t* y, int32_t* idx_out, float* w_out,
                            int32_t* group_out, void* ws, size_t ws_bytes, void* stream);

/*
 * A stack of MoE decoder blocks for the K verify rows, in place:
 *   for l in 0 .. n_layers-1:  x <- x + MoE_l( rmsnorm(x) )
 * (the results of moe_rmsnorm with `eps`, then moe_verify_layer with
 * residual = x and y = x; each layer is one kernel, which applies the
 * RMSNorm itself), all enqueued on `stream` with programmatic overlap
 * between kernels.  All layers share `hidden`.
 *   layers   host array of n_layers layer descriptions (read during the call)
 *   x        bf16 [K][hidden], the residual stream, updated in place
 *   ws       moe_verify_stack_workspace_size(layers, n_layers, K) bytes,
 *            zero-filled before first use
 */
size_t moe_verify_stack_workspace_size(const moe_layer* layers, int n_layers, int K);
moe_status moe_verify_stack(const moe_layer* layers, int n_layers, uint16_t* x, int K, float eps, void* ws,
                            size_t ws_bytes, void* stream);

/*
 * moe_verify_layer without a caller-provided workspace, for callers that
 * cannot allocate device memory: for example an engine whose allocator owns
 * the whole GPU and forbids outside cudaMalloc calls, or a latency-critical
 * decode loop that cannot afford cudaMalloc's implicit device
 * synchronisation.  The pages have no counterpart of this entry point.
 *
 * Same results as moe_verify_layer.  The scratch space (routing tables,
 * intermediate activations, partial sums, counters) is a fixed 8 MiB array
 * compiled into the library; every GPU that loads the library holds it until
 * the process exits.  A call whose layer needs more workspace than that
 * (moe_verify_layer_workspace_size) returns MOE_ERR_WORKSPACE_TOO_SMALL.
 * The inputs and outputs are still the caller's device buffers.
 *  - The call allocates nothing: no cudaMalloc, no cudaFree, no allocating
 *    library routine.
 *  - The first call on a device looks up the array's address on that device
 *    (the device current in the calling thread, which must be the device of
 *    `stream`) and zero-fills it once; make that first call before any
 *    stream capture.
 *  - Every call on a device shares the one array and keeps the last call's
 *    contents (later calls rely on them).  Calls that overlap
 *    on the GPU (different streams, or different host threads) race on the
 *    array and give wrong results: serialise them.
 *  - A device-side wait that runs out of time leaves y undefined and is not
 *    reported by this entry point (use moe_verify_layer with your own
 *    workspace and moe_workspace_error where that matters).
 */
moe_status moe_verify_layer_static(const moe_layer* layer, const uint16_t* x_norm, int K,
                                   const uint16_t* residual, uint16_t* y, int32_t* idx_out, float* w_out,
                                   int32_t* group_out, void* stream);

/*
 * Profiling variant of moe_verify_layer for benchmarks: identical results,
 * but the layer's one kernel is launched without programmatic overlap with
 * its neighbours and, when `events` is not NULL, the cudaEvent_t handles
 * events[0..3] are recorded on `stream`: events 0 and 1 before the kernel
 * (they bracket no work; older layouts had a separate router kernel there)
 * and events 2 and 3 after it, so events 1 -> 2 time the kernel.  Inside a
 * stream capture the events are recorded as external event nodes.
 */
moe_status moe_verify_layer_profiled(const moe_layer* layer, const uint16_t* x_norm, int K,
                                     const uint16_t* residual, uint16_t* y, void* ws, size_t ws_bytes,
                                     void* stream, void* const* events);

/*
 * Accepted prefix of a drafted block: the first i with draft[i] != target[i],
 * or K when all match (README, opening section: decode advances by the
 * longest correct prefix).
 *   draft, target  int32 [K] (may be NULL when K == 0);  n_accepted  int32 [1] out.
 *   0 <= K <= 4096.
 */
moe_status verify_accept_prefix(const int32_t* draft, const int32_t* target, int K,
                                int32_t* n_accepted, void* stream);

/*
 * RMSNorm with unit gain between blocks of the verify step:
 *   out_r = bf16( x_r * 1/sqrt(mean(x_r^2) + eps) )
 * in FP32 in the router's fixed order (its output decides the top-k):
 * the sum of squares is the fixed-order dot product of the row with itself,
 * then one correctly rounded FP32 operation per step.
 *   x, out  bf16 [K][H]; 1 <= K <= 16; H a multiple of 256.
 */
moe_status moe_rmsnorm(const uint16_t* x, int K, int H, float eps, uint16_t* out, void* stream);

/* Bytes of workspace moe_lm_head_argmax needs for K rows (zero-filled once
 * before first use; calls leave it ready for the next call).  Its first
 * int32 is the error word that moe_workspace_error reads (a device-side wait
 * that ran out: MOE_ERR_DEVICE_TIMEOUT). */
size_t moe_lm_head_workspace_size(int K);

/*
 * Greedy token of every verify row (PR #844, "5. Numerical safety": the
 * verifier takes the argmax over every row):
 *   tok_r = argmax_v  x_norm_r . W_v   (FP32, the router's fixed order;
 *                                       an exact tie goes to the lower v)
 *   x_norm bf16 [K][H]; W bf16 [V][H]; tok int32 [K] out;
 *   best_logit float [K] out (nullable): the winning logit.
 *   1 <= K <= 16; H a multiple of 256, at most 2048.
 */
moe_status moe_lm_head_argmax(const uint16_t* x_norm, int K, int H, const uint16_t* W, int V, int32_t* tok,
                              float* best_logit, void* ws, size_t ws_bytes, void* stream);

/*
 * Position handling of an attention block (README, "Why this challenge
 * exists": Laguna alternates three sliding-window layers -- 512-token
 * window, plain RoPE at theta 10000 -- with one full-attention layer per
 * block of four -- YaRN rotary with a 0.5 partial-rotary factor).
 *   window       a row at position p sees positions p - window + 1 .. p
 *                (0: every position); at least 16 when set
 *   rotary_dim   RoPE on the first rotary_dim dims of every q and new-key
 *                head (pairs i, i + rotary_dim/2, "rotate half"), at
 *                positions C .. C+K-1 (C = the valid cache length); 0 = none
 *   rope_theta   RoPE base: pair i turns by p * theta^(-2i/rotary_dim)
 *   yarn_factor  > 1: YaRN frequencies (NTK-by-parts ramp between 1 and 32
 *                rotations over yarn_orig_ctx positions, interpolation by
 *                yarn_factor below it) and logits scaled by
 *                (0.1 ln yarn_factor + 1)^2; <= 1: plain RoPE
 * The cached keys are taken as already rotated (a cache stores rotated keys).
 */
typedef struct {
  int window;
  int rotary_dim;
  float rope_theta;
  float yarn_factor;
  int yarn_orig_ctx;
} moe_attn_pos;

/*
 * GQA attention block of the verify step (README, "Why this challenge
 * exists": GQA with 8 KV heads at head_dim 128; the verify forward runs all
 * K drafted rows at once):
 *   xn = rmsnorm(x)  (as moe_rmsnorm)
 *   q = bf16(xn . Wq^T), k_new = bf16(xn . Wk^T), v_new = bf16(xn . Wv^T)
 *   o[r, h] = bf16( softmax_p( q[r,h] . key_p / sqrt(128) ) . value_p )
 *             over the cached positions of KV head h / (nq/nkv) and the
 *             new positions 0..r (block-causal)
 *   x_out = bf16( x + o . Wo^T )
 *   x, x_out bf16 [K][H] (x_out may alias x); Wq [nq*128][H], Wk, Wv
 *   [nkv*128][H], Wo [H][nq*128]; kcache, vcache [nkv][C][128];
 *   kv_len: NULL -- all C cached positions are valid and the caches are
 *     only read; or a device int32: *kv_len of the C positions are valid
 *     and the K new keys and values are written into the caches in place at
 *     positions *kv_len .. *kv_len + K - 1 (the caches then hold C positions
 *     of capacity; an append past C is refused and recorded as
 *     MOE_ERR_CAPACITY in the workspace error word).  The length itself is
 *     not changed here: moe_kv_commit counts the accepted rows in.
 *   pos: NULL, or the window / rotary embedding of the block (moe_attn_pos).
 *   k_new_out, v_new_out: optional [K][nkv*128] copies of the new (rotated)
 *   keys and values; o_out: optional [K][nq*128] copy of the attention
 *   output o (before the o-projection).
 * Envelope: head_dim 128, nq even, nq % nkv == 0, K * nq/nkv <= 64, H a
 * multiple of 256 up to 4096, nq*128 <= 8192, K * nq <= 768, C a multiple
 * of 16.
 */
size_t moe_attention_workspace_size(int K, int H, int nq, int nkv, int head_dim);
moe_status moe_attention_block(const uint16_t* x, int K, int H, int nq, int nkv, int head_dim, int C,
                               const uint16_t* Wq, const uint16_t* Wk, const uint16_t* Wv, const uint16_t* Wo,
                               uint16_t* kcache, uint16_t* vcache, const int32_t* kv_len, const moe_attn_pos* pos,
                               float eps, uint16_t* x_out, uint16_t* k_new_out, uint16_t* v_new_out,
                               uint16_t* o_out, void* ws, size_t ws_bytes, void* stream);

/*
 * The dense SwiGLU MLP block of Laguna's layer 0 (README, "Why this
 * challenge exists": layer 0 has a dense MLP, intermediate 8192, bf16):
 *   xn = rmsnorm(x);  h = bf16( silu(xn . Wg^T) * (xn . Wu^T) )
 *   x_out = bf16( x + h . Wd^T )      (FP32 accumulation)
 *   x, x_out bf16 [K][H] (may alias); Wg, Wu [I][H]; Wd [H][I]; I a
 *   multiple of 256, K * I <= 98304.
 */
size_t moe_dense_mlp_workspace_size(int K, int H, int I);
moe_status moe_dense_mlp_block(const uint16_t* x, int K, int H, int I, const uint16_t* Wg, const uint16_t* Wu,
                               const uint16_t* Wd, float eps, uint16_t* x_out, void* ws, size_t ws_bytes,
                               void* stream);

/*
 * The full verify step of a decoder with GQA attention and MoE blocks:
 *   for each layer l:  x <- attention_block_l(x)          (moe_attention_block)
 *                      x <- x + MoE_l(rmsnorm(x))          (moe_verify_stack)
 *   target_r = argmax_v rmsnorm(x)_r . lm_head_v           (moe_lm_head_argmax)
 *   n_accepted = first r with draft_r != target_r, else K (verify_accept_prefix)
 * i.e. one target forward over the K drafted rows, its greedy token per row,
 * and how far decode advances (README, opening section and "Why this
 * challenge exists"; PR #844, "5. Numerical safety": argmax over every row).
 */
typedef struct {
  const uint16_t *Wq, *Wk, *Wv, *Wo;  /* bf16 attention projections (see moe_attention_block) */
  uint16_t *kcache, *vcache;          /* bf16 [nkv][ctx][128] */
  moe_layer moe;                      /* the MoE block of the layer */
  int n_q_heads;                      /* 0: the model's n_q_heads */
  moe_attn_pos pos;                   /* all zero: no window, no rotary embedding */
  const uint16_t *mlp_gate, *mlp_up, *mlp_down;  /* non-NULL: a dense SwiGLU MLP block
                                         (moe_dense_mlp_block, intermediate mlp_inter)
                                         instead of the MoE block */
  int mlp_inter;
} moe_decoder_layer;

typedef struct {
  int n_layers, hidden, n_q_heads, n_kv_heads, head_dim, ctx, vocab;
  float eps;                          /* RMSNorm epsilon */
  const moe_decoder_layer* layers;    /* host array of n_layers (read during the call) */
  const uint16_t* lm_head;            /* bf16 [vocab][hidden] */
  const int32_t* kv_len;              /* NULL: every layer attends over all ctx cached positions,
                                         caches read only; else a device int32 shared by the
                                         layers: ctx is the caches' capacity, *kv_len positions
                                         are valid, and each step appends its K rows' keys and
                                         values in place (see moe_attention_block) */
} moe_verify_model;

size_t moe_verify_step_workspace_size(const moe_verify_model* model, int K);

/*   x          bf16 [K][hidden]: the rows' input to layer 0; overwritten with
 *              the final residual stream
 *   draft      int32 [K] drafted tokens;  target int32 [K] out;  n_accepted int32 [1] out
 *   ws         moe_verify_step_workspace_size bytes, zero-filled before first use */
moe_status moe_verify_step(const moe_verify_model* model, uint16_t* x, int K, const int32_t* draft,
                           int32_t* target, int32_t* n_accepted, void* ws, size_t ws_bytes, void* stream);

/*
 * The multi-round verify loop with an in-place KV cache (PR #844, "8. What I
 * looked at and did NOT ship", items 1 and 2, and "10. Next step": keep the
 * verify rows' keys and values in a temporally ordered arena and drop the
 * rejected rows by trimming, with no snapshot and no replay forward).
 *
 * moe_kv_commit: after a step of K rows with n accepted drafts, rows
 * 0 .. min(n + 1, K) - 1 hold committed tokens (row 0 the last committed
 * token, row i + 1 the draft the target confirmed at row i), so
 *   *kv_len += min(*n_accepted + 1, K)   (clamped to `capacity`)
 * Their keys and values were already appended in place by the step; the
 * other rows' entries lie past the new length and are overwritten by the
 * next step.  One device thread; nothing is copied.
 */
moe_status moe_kv_commit(int32_t* kv_len, const int32_t* n_accepted, int K, int capacity, void* stream);

/*
 * A drafter with a controlled acceptance rate, for benchmarks and tests: no
 * draft model, the drafts are made from the target's own greedy tokens:
 *   draft_r = target_r                          if coin[r] != 0
 *           = (target_r + 1 + alt[r]) mod vocab otherwise (never target_r)
 *   target, alt int32 [K] (0 <= alt[r] < vocab - 1); coin uint8 [K]; draft int32 [K] out.
 * (The verify rows are synthetic activations, so the drafts do not feed the
 * forward; they only decide how far each round advances.)
 */
moe_status moe_synthetic_drafts(const int32_t* target, const uint8_t* coin, const int32_t* alt, int K, int vocab,
                                int32_t* draft, void* stream);

/*
 * R verify rounds on the device, one after the other, with no host
 * involvement between them: for round t
 *   x_work <- x_rounds[t];  forward (every layer appends its K rows' keys and
 *   values in place at *kv_len ..);  targets[t] = greedy tokens;
 *   drafts[t] = moe_synthetic_drafts(targets[t], coin[t], alt[t]);
 *   n_accepted[t] = accepted prefix;  moe_kv_commit.
 *   model->kv_len must be set; x_rounds bf16 [R][K][hidden]; coin uint8
 *   [R][K]; alt int32 [R][K]; x_work bf16 [K][hidden]; targets, drafts int32
 *   [R][K] out; n_accepted int32 [R] out; ws as moe_verify_step.
 * A round whose append would pass the capacity records MOE_ERR_CAPACITY.
 */
moe_status moe_verify_rounds(const moe_verify_model* model, const uint16_t* x_rounds, int R, int K, const uint8_t* coin,
                             const int32_t* alt, uint16_t* x_work, int32_t* targets, int32_t* drafts,
                             int32_t* n_accepted, void* ws, size_t ws_bytes, void* stream);

/*
 * Reads the device error word of a workspace (0 = none, else a negative
 * moe_status) and clears it.  Synchronises `stream`.
 */
moe_status moe_workspace_error(void* ws, int* code, void* stream);

/* A short English description of a status. */
const char* moe_status_string(moe_status s);

/*
 * The address by which the device reaches page-locked host memory (pinned
 * with cudaHostAlloc or cudaHostRegister and mapped, as every pinned buffer
 * is under unified addressing).  The activations of a layer call -- x_norm,
 * residual and y of moe_verify_layer -- may be such memory, and a caller's
 * host buffers then take part in the call with no copy of their own: rows in
 * host memory are staged once into the workspace by the call's first kernel
 * (their loads overlap the previous kernel on the stream), the residual is
 * read and y written across the host link directly.
 * (Weights, caches and workspaces must be device memory.)  Returns
 * MOE_ERR_INVALID_ARG, with *dev untouched, when `host` is not mapped
 * page-locked memory -- also for pageable memory on a system whose device
 * could reach it; a layer call refuses activations in pageable memory with
 * MOE_ERR_INVALID_ARG.
 */
moe_status moe_host_pointer(const void* host, void** dev);

/*
 * Test hook: upper bound, in nanoseconds, of every device-side wait in
 * kernels launched after this call (default 2e9).  0 makes every wait give
 * up at once, which exercises the timeout path without hanging a GPU.
 */
void moe_debug_set_wait_limit_ns(uint64_t ns);

/*
 * Test hook: byte offset, inside a moe_verify_layer workspace, of the down
 * partials d_{r,s} the combine reads: [K][top_k + 1][hidden] 64-bit words
 * whose low 32 bits are the FP32 partial (slot top_k = the shared expert);
 * they hold the last call's values.  0 on an invalid layer or K.
 */
size_t moe_debug_partials_offset(const moe_layer* layer, int K);

/*
 * Profiling hook: when `buf` (device memory, one row of 80 uint64 per SM)
 * is not NULL, experts kernels launched afterwards record %globaltimer
 * stamps of their milestones in it (NULL turns it off).
 */
void moe_debug_set_trace(void* buf);

#ifdef __cplusplus
}
#endif

#endif /* MOE_VERIFY_H */
