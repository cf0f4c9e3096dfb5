/*
 * mlora.h -- C ABI of libmlora.so: one multi-tenant LoRA training step
 * (forward_backward + optim_step) over a mixed batch whose tokens belong to
 * many LoRA adapters that share one frozen base, on one sm_103a GPU.
 *
 * The model.  A token embedding E [V x d]; L residual blocks
 *     u = W1 h + gamma_a B1_a (A1_a h),   act = silu(u),
 *     h <- h + W2 act + gamma_a B2_a (A2_a act)
 * with W1 [f x d], W2 [d x f] frozen and shared, and per adapter a and layer
 * l the trainable factors A1 [r x d], B1 [f x r], A2 [r x f], B2 [d x r],
 * gamma_a = alpha_a / r_a (Deep Dive - Tinker, "LoRA is the adaptation
 * boundary": W' = W + gamma B A); then an untied LM head Wout [V x d] and the
 * target-token logprob l_t = z[y_t] - logsumexp(z), z = Wout h (Tinker API
 * Implementation on TPUs, section 10.3-10.4: the [tokens x vocab] logits are
 * never stored whole).  The LM-head backward runs in chunks of at most 16,384
 * rows and has two modes (mlora_set_lm_backward): by default it recomputes
 * each chunk's logits with a second GEMM, as that section describes; on
 * request it instead keeps each chunk's logits from the forward in a bounded
 * buffer and reads them back.
 *
 * Conventions for every entry point:
 *  - Return value: MLORA_OK (0) or a negative MLORA_E_* code; the message of
 *    the last failure on the calling thread is mlora_last_error().
 *  - "device" pointers are CUDA device memory of the current device; "host"
 *    pointers are ordinary host memory.  The caller owns every buffer it
 *    passes; the library owns every buffer it allocates (freed by
 *    mlora_destroy).  The library never keeps a caller pointer after a call
 *    returns.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Work is queued asynchronously on it; calls on one handle must
 *    be serialised by the caller (one training client, ordered requests:
 *    Deep Dive - Tinker, "optim_step advances adapter state").
 *  - Errors found on the device (token id >= V, target >= V, adapter id >=
 *    n_adapters) never trap: the kernels skip the offending token, write NaN
 *    as its logprob, and raise a status bit that mlora_check_status() reports
 *    as MLORA_E_RANGE.  A device wait that exceeds its bound sets
 *    MLORA_E_TIMEOUT the same way.
 */
#ifndef MLORA_H
#define MLORA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Routing tile height: every adapter's segment of the sorted token matrix is
 * padded to a multiple of this many rows, so that no GEMM row tile mixes two
 * adapters (tinker-ticks, "How the SGMV kernel works": segment indices over
 * the flattened tokens). */
#define MLORA_TILE_M 128
/* Largest supported LoRA rank; ranks must also be multiples of 4. */
#define MLORA_MAX_RANK 64

enum {
    MLORA_OK = 0,
    MLORA_E_ARG = -1,      /* invalid argument or configuration              */
    MLORA_E_RANGE = -2,    /* device saw an id out of range (token/adapter)  */
    MLORA_E_CUDA = -3,     /* a CUDA runtime call failed                     */
    MLORA_E_NOMEM = -4,    /* device allocation failed                       */
    MLORA_E_TIMEOUT = -5,  /* a bounded device wait gave up                  */
    MLORA_E_IO = -6,       /* file write failed (save_state)                 */
    MLORA_E_UNSUPPORTED = -7 /* no sm_103a device / feature missing          */
};

typedef enum { MLORA_BF16 = 0, MLORA_FP32 = 1 } mlora_dtype;

/* Loss kinds (Deep Dive - Tinker, "The RL datum shape"); every loss is a sum
 * over tokens with no normalisation.
 *   CROSS_ENTROPY        L = -sum_t w_t l_t
 *   IMPORTANCE_SAMPLING  L = -sum_t r_t A_t,             r_t = exp(l_t - s_t)
 *   PPO                  L = -sum_t min(r_t A_t, clip(r_t, 1-eps, 1+eps) A_t)
 * A token whose inputs, logprob or ratio are not finite contributes neither
 * value nor gradient (Tinker API Implementation on TPUs, section 12). */
typedef enum {
    MLORA_CROSS_ENTROPY = 0,
    MLORA_IMPORTANCE_SAMPLING = 1,
    MLORA_PPO = 2
} mlora_loss;

/* Selector for mlora_read_adapter / mlora_write_adapter.  Shapes (row-major,
 * fp32): A1 [r x d], B1 [f x r], A2 [r x f], B2 [d x r].  GRAD_* are the
 * accumulated gradients, M_* / V_* the Adam moments. */
typedef enum {
    MLORA_A1 = 0, MLORA_B1 = 1, MLORA_A2 = 2, MLORA_B2 = 3,
    MLORA_GRAD_A1 = 4, MLORA_GRAD_B1 = 5, MLORA_GRAD_A2 = 6, MLORA_GRAD_B2 = 7,
    MLORA_M_A1 = 8, MLORA_M_B1 = 9, MLORA_M_A2 = 10, MLORA_M_B2 = 11,
    MLORA_V_A1 = 12, MLORA_V_B1 = 13, MLORA_V_A2 = 14, MLORA_V_B2 = 15
} mlora_tensor;

typedef struct mlora mlora_t;

typedef struct {
    int32_t vocab;         /* V                                              */
    int32_t d_model;       /* d, multiple of 64                              */
    int32_t d_ffn;         /* f, multiple of 64                              */
    int32_t n_layers;      /* L >= 1                                         */
    int32_t dtype;         /* mlora_dtype of the frozen base and activations */
    int32_t n_adapters;    /* 1 .. 1024                                      */
    const int32_t* ranks;  /* host [n_adapters]; 1..MLORA_MAX_RANK, % 4 == 0 */
    const float* alphas;   /* host [n_adapters]; gamma_a = alphas[a]/ranks[a] */
    int64_t max_tokens;    /* largest n_tokens any call will pass (>= 1)     */
} mlora_config;

/* Initial values, all DEVICE pointers, read once by mlora_create and copied
 * into library-owned memory.  Base tensors hold `dtype` elements (bf16 as
 * raw 16-bit patterns).  Adapter arrays are HOST arrays of n_adapters *
 * n_layers device pointers to fp32 tensors, indexed [a * n_layers + l]; a NULL
 * array or a NULL entry initialises that tensor to zero. */
typedef struct {
    const void* E;                 /* [V x d]                  */
    const void* const* W1;         /* host [n_layers] -> [f x d] */
    const void* const* W2;         /* host [n_layers] -> [d x f] */
    const void* Wout;              /* [V x d]                  */
    const float* const* A1;
    const float* const* B1;
    const float* const* A2;
    const float* const* B2;
} mlora_init;

/* A flattened token batch: DEVICE int32 arrays of length n_tokens.  Token t
 * has input id tokens[t], target id targets[t] (the next token of its
 * sequence) and adapter adapter_ids[t]. */
typedef struct {
    int64_t n_tokens;              /* 0 .. max_tokens */
    const int32_t* tokens;
    const int32_t* targets;
    const int32_t* adapter_ids;
} mlora_batch;

/* Per-token loss inputs, DEVICE fp32 arrays of length n_tokens (those the
 * loss kind does not read may be NULL). */
typedef struct {
    const float* weights;           /* CROSS_ENTROPY: w_t                 */
    const float* advantages;        /* IMPORTANCE_SAMPLING / PPO: A_t      */
    const float* sampler_logprobs;  /* IMPORTANCE_SAMPLING / PPO: s_t      */
    float clip_eps;                 /* PPO clip range eps                 */
} mlora_loss_inputs;

/* Adam hyper-parameters (Deep Dive - Tinker, "optim_step advances adapter
 * state": AdamW-equivalent, default weight decay 0).  Update per element:
 *   m = b1 m + (1-b1) G;  v = b2 v + (1-b2) G^2;  t = t + 1
 *   p = p - lr * ( (m / (1-b1^t)) / (sqrt(v / (1-b2^t)) + eps) + wd * p ) */
typedef struct {
    float lr, beta1, beta2, eps, weight_decay;
} mlora_adam;

/* Create a handle: validates the config, allocates all device memory for up
 * to max_tokens tokens, copies the base and the initial adapters, zeroes
 * gradients and moments, sets every adapter's step count to 0.  Synchronous.
 * Errors: E_ARG (bad config/NULL), E_NOMEM, E_CUDA, E_UNSUPPORTED (a BF16
 * handle needs an sm_103 device). */
int mlora_create(const mlora_config* cfg, const mlora_init* init, mlora_t** out);

/* Free everything the handle owns (synchronises the device first). */
int mlora_destroy(mlora_t* h);

/* Target-token logprobs of every token (no gradient, no state change).
 * logprobs_out: DEVICE fp32 [n_tokens], caller-owned. */
int mlora_forward(mlora_t* h, const mlora_batch* b, float* logprobs_out, void* stream);

/* Forward, loss and adapter-only backward.  Gradients ACCUMULATE into the
 * handle's per-adapter buffers until mlora_optim_step consumes them; every
 * adapter with at least one token is marked as touched.
 * logprobs_out: DEVICE fp32 [n_tokens] (may be NULL).
 * loss_out: DEVICE fp64 [n_adapters] (may be NULL): loss summed over each
 * adapter's tokens of this call. */
int mlora_forward_backward(mlora_t* h, const mlora_batch* b, int32_t loss_kind,
                           const mlora_loss_inputs* li, float* logprobs_out,
                           double* loss_out, void* stream);

/* Backpropagate the surrogate sum_t g_t l_t with the caller's
 * g_t = dC/dl_t (Deep Dive - Tinker, "The RL datum shape"; the Telegram note
 * on forward_backward_custom: the server re-runs the forward and backprops
 * sum(logprobs * dLoss/dLogprobs)).  dloss_dlogprobs: DEVICE fp32 [n_tokens].
 * Outputs and accumulation as mlora_forward_backward (loss_out receives
 * sum_t g_t l_t per adapter). */
int mlora_forward_backward_custom(mlora_t* h, const mlora_batch* b,
                                  const float* dloss_dlogprobs, float* logprobs_out,
                                  double* loss_out, void* stream);

/* One Adam step per selected adapter, consuming (and zeroing) its gradient.
 * adapters: HOST int32 [n] of adapter ids, or NULL to select every adapter
 * touched since the previous optim_step.  An adapter whose accumulated
 * gradient holds a non-finite value keeps its weights, moments and step
 * count; its gradient is still consumed and skipped_out[a] is set to 1
 * (Tinker API Implementation on TPUs, section 12: non-finite optimizer
 * updates are skipped).  skipped_out: DEVICE int32 [n_adapters] (may be
 * NULL), 0 for every adapter not skipped. */
int mlora_optim_step(mlora_t* h, const mlora_adam* p, const int32_t* adapters,
                     int32_t n, int32_t* skipped_out, void* stream);

/* Write a checkpoint of every adapter (weights and Adam state) to `path`.
 * Synchronises `stream`.  Format, little-endian: 8-byte magic "MLORASTA",
 * u32 version = 1, u32 n_adapters, u32 n_layers, u32 d_model, u32 d_ffn,
 * u32 0; then per adapter: u32 rank, f32 alpha, u64 step count, followed by
 * the weights, the first moments and the second moments, each as, for every
 * layer, A1, B1, A2, B2 in fp32 row-major.  (Deep Dive - Tinker, "save_state
 * creates a recovery point".)  Errors: E_IO, E_CUDA. */
int mlora_save_state(mlora_t* h, const char* path, void* stream);

/* Restore every adapter from a checkpoint written by mlora_save_state
 * (Deep Dive - Tinker, "optim_step advances adapter state" and "save_state
 * creates a recovery point": loading weights alone resets the optimizer
 * history; loading with the optimizer restores the saved moments).
 * with_optimizer = 0 (load_state): weights from the file; first and second
 * moments and step counts set to zero, so the next Adam step of each adapter
 * is its first.  with_optimizer = 1 (load_state_with_optimizer): weights,
 * moments and step counts from the file.  In both cases any gradient
 * accumulated before the call is discarded (with its touched and non-finite
 * flags), and the padded-rank copies the GEMMs read are refreshed.
 * The file must match the handle: adapter count, n_layers, d_model, d_ffn,
 * and per adapter rank and alpha (else E_ARG).  E_IO: cannot open, wrong
 * magic or version, truncated, or trailing bytes.  The file is read and
 * checked in full before the handle changes: on any error the adapter state
 * is untouched.  Synchronises `stream` before and after the upload. */
int mlora_load_state(mlora_t* h, const char* path, int32_t with_optimizer, void* stream);

/* Export one adapted projection as a standalone base matrix (Deep Dive -
 * Tinker, "Checkpoints and export paths": merging W' = W + gamma B A turns
 * an adapter into a standalone model; gamma = alpha / r).
 * which = 0: out = W1[layer] + gamma B1 A1, [d_ffn x d_model];
 * which = 1: out = W2[layer] + gamma B2 A2, [d_model x d_ffn];
 * row-major in the base dtype, out a DEVICE buffer (16-byte aligned) owned
 * by the caller.  B A is taken from the adapter's fp32 master weights: on a
 * bf16 base each factor is split into two bf16 parts so that the tensor-core
 * product carries about 16 significant bits before the single rounding of
 * W + gamma B A to bf16.  A model whose every W1, W2 is replaced by its
 * export and that runs without the adapter gives the adapter's logprobs.
 * Queued on `stream`.  Errors: E_ARG (NULL, unaligned out, adapter, layer
 * or which out of range), E_CUDA. */
int mlora_export_merged(mlora_t* h, int32_t adapter, int32_t layer, int32_t which, void* out,
                        void* stream);

/* ------------------------------------------------------------------------
 * Sampler side: scoring and one-token decode with pinned adapter snapshots
 * (OpenTinker, "Multi-LoRA rollout": rows are batched by pinned adapter
 * version over the shared base projection; tinker-ticks, "Why RL needs
 * batch-invariant kernels": rollout and training logprobs must agree).
 *
 * A sampler shares the frozen base of a training handle (which must outlive
 * it) and holds n_slots adapter snapshots.  Rows stay in batch order, each
 * naming a slot; there is no per-adapter padding.  Every layer runs the
 * training forward's kernels on the same operand values, with each row's
 * adapter applied as its slot's block of a K extension whose other blocks
 * are zero for that row, so a row's logprob is bitwise the one
 * mlora_forward returns for the same token, target and adapter weights.
 * ------------------------------------------------------------------------ */
typedef struct mlora_sampler mlora_sampler_t;
#define MLORA_SAMPLER_MAX_SLOTS 64
#define MLORA_SAMPLER_MAX_ROWS 32768

/* Create a sampler over `trainer`'s frozen base with n_slots (1..64) empty
 * slots and room for max_rows (1..32768) rows per call.  Device memory:
 * per layer 2 * n_slots * 64 * (d + f) base-dtype elements of snapshots,
 * plus per row about 4 * Vpad bytes of kept logits and the activations of
 * one forward.  Errors: E_ARG, E_NOMEM, E_CUDA. */
int mlora_sampler_create(mlora_t* trainer, int32_t n_slots, int64_t max_rows,
                         mlora_sampler_t** out);
int mlora_sampler_destroy(mlora_sampler_t* s);

/* Publish: copy `adapter`'s current weights (every layer's padded-rank
 * base-dtype copies the GEMMs read, and its gamma) from the trainer into
 * `slot`.  The slot keeps them until it is published again, whatever the
 * trainer does meanwhile.  version_out (HOST, may be NULL) receives the
 * adapter's optimizer step count at publication.  Synchronises `stream`.
 * Errors: E_ARG (slot or adapter out of range), E_CUDA. */
int mlora_sampler_publish(mlora_sampler_t* s, int32_t slot, int32_t adapter,
                          int64_t* version_out, void* stream);

/* Score: logprobs_out[t] = log softmax(z_t)[targets[t]] for row t computed
 * with slot slots[t] (compute_logprobs / prefill).  tokens, targets, slots:
 * DEVICE int32 [n]; logprobs_out: DEVICE fp32 [n].  A row whose token,
 * target or slot is out of range or whose slot is unpublished gets NaN and
 * raises the sampler's status bit (mlora_sampler_check_status -> E_RANGE).
 * 0 <= n <= max_rows (else E_ARG).  Queued on `stream`. */
int mlora_sampler_logprobs(mlora_sampler_t* s, const int32_t* tokens, const int32_t* targets,
                           const int32_t* slots, int64_t n, float* logprobs_out, void* stream);

/* One decode step: for row t, the next token is the smallest vocabulary id
 * v with CDF(v) > uniforms[t], CDF the cumulative softmax of the row's
 * logits in vocabulary order (inverse-CDF sampling at temperature 1; the
 * caller draws the uniforms in [0, 1)); logprob_out[t] is that token's
 * logprob, bitwise what mlora_sampler_logprobs returns for it as target.
 * When rounding leaves the cumulative sum at or below u the last token with
 * a non-zero probability is taken.  tokens, slots: DEVICE int32 [n];
 * uniforms: DEVICE fp32 [n]; next_out: DEVICE int32 [n] (-1 for a bad row);
 * logprob_out: DEVICE fp32 [n] (NaN for a bad row).  Queued on `stream`. */
int mlora_sampler_sample(mlora_sampler_t* s, const int32_t* tokens, const int32_t* slots,
                         const float* uniforms, int64_t n, int32_t* next_out, float* logprob_out,
                         void* stream);

/* Synchronise `stream`, return and clear the sampler's status word. */
int mlora_sampler_check_status(mlora_sampler_t* s, void* stream);
int64_t mlora_sampler_kernel_launches(const mlora_sampler_t* s);

/* Copy one fp32 adapter tensor (see mlora_tensor) of adapter `adapter`,
 * layer `layer` into dst (DEVICE, caller-owned, shape as documented there).
 * Test and inspection hook. */
int mlora_read_adapter(mlora_t* h, int32_t adapter, int32_t layer, int32_t which,
                       float* dst, void* stream);

/* Overwrite a weight tensor (MLORA_A1..MLORA_B2 only) from src (DEVICE fp32)
 * and refresh its bf16 copy used by the GEMMs. */
int mlora_write_adapter(mlora_t* h, int32_t adapter, int32_t layer, int32_t which,
                        const float* src, void* stream);

/* Step counts: HOST int64 [n_adapters] out (synchronises `stream`). */
int mlora_get_steps(mlora_t* h, int64_t* steps_out, void* stream);

/* The routing that forward / forward_backward use, exposed for checking:
 * adapter_ids: DEVICE int32 [n]; outputs are DEVICE int32:
 *   perm[n]              stable order of token positions grouped by adapter
 *   seg_off[n_adapters+1] exclusive prefix of per-adapter token counts
 *   pad_off[n_adapters+1] the same with each segment padded to MLORA_TILE_M
 *   tile_ad[n / MLORA_TILE_M + n_adapters + 1] adapter of each padded row
 *                        tile, -1 after the last tile
 * Ids out of range are left out and raise MLORA_E_RANGE on check_status. */
int mlora_get_routing(mlora_t* h, const int32_t* adapter_ids, int64_t n, int32_t* perm,
                      int32_t* seg_off, int32_t* pad_off, int32_t* tile_ad, void* stream);

/* Routing without allocation.  The same stable grouping as
 * mlora_get_routing (same outputs, same layout, same -1 tail of tile_ad), but
 * with no handle and no device allocation of any kind: for callers that
 * cannot call cudaMalloc -- their device memory is owned by another
 * allocator, or their loop must not pay for cudaMalloc's possible device
 * synchronisation.  The pages have no counterpart of this entry point; it
 * exists for such embedders.
 *   adapter_ids: DEVICE int32 [n]; n <= MLORA_NOALLOC_MAX_TOKENS
 *   n_adapters:  1 .. MLORA_NOALLOC_MAX_ADAPTERS
 *   perm, seg_off, pad_off, tile_ad: DEVICE int32 outputs sized as for
 *   mlora_get_routing.
 * Scratch lives in a fixed array inside the library (about 0.6 MB per GPU,
 * held until the process exits).  The first call on a device resolves that
 * array's device address (cudaGetSymbolAddress) with the device current.
 * All calls share the array: calls whose GPU work may overlap race and must
 * be ordered by the caller.  Ids out of range are left out, as in
 * mlora_get_routing, but are not reported (there is no handle status word).
 * Errors: E_ARG for sizes beyond the limits or NULL pointers, E_CUDA. */
#define MLORA_NOALLOC_MAX_TOKENS 65536
#define MLORA_NOALLOC_MAX_ADAPTERS 128
int mlora_routing_noalloc(const int32_t* adapter_ids, int64_t n, int32_t n_adapters,
                          int32_t* perm, int32_t* seg_off, int32_t* pad_off, int32_t* tile_ad,
                          void* stream);

/* Deterministic (batch-invariant) mode (tinker-ticks, "Why RL needs
 * batch-invariant kernels": a token's result must not depend on how many
 * other tokens share the batch, and must repeat bit for bit).
 *
 * Logprobs and losses are batch-invariant in both modes: every GEMM's tile
 * shape and instruction depend only on the layer widths, each output element
 * sums its contraction in one fixed order inside one tile, the LM-head
 * log-sum-exp merges its column-tile partials in a fixed order, and each
 * adapter's loss sum runs over its own padded segment.  What on = 1 adds is
 * the gradients: each adapter's token rows form ONE gradient work chunk
 * (instead of chunks of 1024 padded rows met by fp32 atomics in arrival
 * order), so every gradient element has one writer and one summation order.
 * An adapter's gradients, and the weights after mlora_optim_step, are then
 * bitwise the same on every run and whichever other adapters share the
 * batch (given its own tokens in the same order).  Cost: an adapter with
 * many tokens reduces over them in fewer, longer tiles.
 * The mode is a host-side flag read at each forward/backward launch; the
 * default is 0.  Errors: E_ARG (NULL handle, on not 0 or 1). */
int mlora_set_deterministic(mlora_t* h, int32_t on);

/* How the LM-head backward obtains each row chunk's logits (Tinker API
 * Implementation on TPUs, section 10.4: fused linear cross-entropy, whose
 * custom backward keeps only the hidden rows and recomputes one tile of
 * logits at a time).  Both modes first run the LM-head forward and the loss
 * epilogue, then walk the rows in chunks of at most 16,384:
 *   MLORA_LM_RECOMPUTE (the default of a new handle): a second LM-head GEMM
 *     over the chunk recomputes its logits and its epilogue writes
 *     dz = g (onehot(y) - softmax(z)) into a bf16 chunk buffer, then
 *     dh = dz Wout.  Extra device memory: one dz chunk buffer
 *     (16,384 x Vpad base-dtype elements, 5 GB at V = 151,936 in bf16).
 *   MLORA_LM_KEEP_LOGITS: the forward GEMM of each chunk also stores its
 *     logits; an elementwise pass turns them into dz on a side stream while
 *     the next chunk's GEMMs run.  Saves the recompute GEMM (2 N V d FLOPs per
 *     step) for two kept-logit chunk buffers and a second dz buffer (15 GB
 *     more at V = 151,936 in bf16).  A bf16 handle keeps, per 256-column
 *     tile of a row, e = exp(z - m) in fp16 with the tile's maximum m (a
 *     float per row and tile), and forms dz = g (onehot(y) - e exp(m - lse));
 *     an fp32 handle keeps the fp32 logits.
 * Both modes give bitwise the same logprobs, losses and gradients: the
 * recomputed accumulator is the forward's, and dz is formed by the same
 * arithmetic (on a bf16 handle the recompute epilogue forms the same fp16 e).  Selecting KEEP_LOGITS allocates its buffers (E_NOMEM if they do
 * not fit; the handle then stays in RECOMPUTE); selecting RECOMPUTE frees
 * them.  Synchronises the device.  Errors: E_ARG (NULL handle, unknown mode),
 * E_NOMEM, E_CUDA. */
enum { MLORA_LM_RECOMPUTE = 0, MLORA_LM_KEEP_LOGITS = 1 };
int mlora_set_lm_backward(mlora_t* h, int32_t mode);

/* Synchronise `stream`, then return and clear the device status word:
 * MLORA_OK, MLORA_E_RANGE or MLORA_E_TIMEOUT. */
int mlora_check_status(mlora_t* h, void* stream);

/* Per-kernel-class timing for measurement.  While enabled, the library
 * brackets each of its kernel launches with CUDA events recorded on the
 * launch stream and tags it with one of the MLORA_PROF_* classes below.
 * mlora_profile_read synchronises those events and returns, per class, the
 * accumulated milliseconds and launch counts since the last reset
 * (ms_out / launches_out: HOST arrays of MLORA_PROF_CLASSES entries).
 * MLORA_PROF_LM_DZ times how the LM-head backward forms dz: the elementwise
 * pass over kept logits, or the recompute GEMM in the default mode.
 * Enabling costs two event records per launch. */
enum {
    MLORA_PROF_ROUTING = 0, MLORA_PROF_EMBED = 1, MLORA_PROF_SHRINK = 2,
    MLORA_PROF_W1_FWD = 3, MLORA_PROF_W2_FWD = 4, MLORA_PROF_LM_FWD = 5,
    MLORA_PROF_LOSS = 6, MLORA_PROF_LM_DZ = 7, MLORA_PROF_LM_DH = 8,
    MLORA_PROF_W2_BWD = 9, MLORA_PROF_W1_BWD = 10, MLORA_PROF_GRAD = 11,
    MLORA_PROF_ADAM = 12, MLORA_PROF_OTHER = 13, MLORA_PROF_CLASSES = 14
};
int mlora_profile_enable(mlora_t* h, int32_t on);
int mlora_profile_read(mlora_t* h, double* ms_out, int64_t* launches_out, int32_t reset);

/* Number of kernels this handle has launched so far. */
int64_t mlora_kernel_launches(const mlora_t* h);

/* Bytes of device memory the handle owns. */
int64_t mlora_device_bytes(const mlora_t* h);

/* Message of the last failure on the calling thread ("" if none). */
const char* mlora_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* MLORA_H */
