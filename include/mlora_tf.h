/*
 * mlora_tf.h -- C ABI of libmlora.so for the transformer-block model: the same
 * multi-tenant LoRA step (forward_backward + optim_step over a mixed batch of
 * many adapters sharing one frozen base) with the pages' real layer shape.
 *
 * The model.  tinker-ticks, "How the SGMV kernel works": LoRA rides on every
 * linear projection of a layer -- q, k, v, o around attention and gate, up,
 * down in the MLP, seven per layer; attention itself is not adapted.  Per
 * layer l, with RMSNorm(x) = x / sqrt(mean(x^2) + eps) * g (frozen gain g):
 *     x = RMSNorm_attn(h);  q, k, v = P_q(x), P_k(x), P_v(x)
 *     q, k = rope(q), rope(k);  o = causal attention inside each sequence
 *     h = h + P_o(o);  x = RMSNorm_mlp(h);  h = h + P_down(silu(P_gate x) * P_up x)
 * where P_p(x) = W_p x + gamma_a B_p,a (A_p,a x) for the token's adapter a
 * (Deep Dive - Tinker, "LoRA is the adaptation boundary": W' = W + gamma B A,
 * gamma = alpha / r).  Then z = Wout RMSNorm_final(h) and the target logprob
 * l = z[y] - logsumexp(z) (Tinker API Implementation on TPUs, section 10.3),
 * with the [tokens x vocab] logits never stored whole.
 * Attention: n_heads query heads and n_kv_heads key/value heads of width
 * head_dim = 128; query head j reads key/value head j / (n_heads/n_kv_heads);
 * scores are scaled by 1/sqrt(128).  Rotary embedding: for i < 64 the pair
 * (x_i, x_{i+64}) of each q and k head is rotated by pos * theta^(-i/64).
 *
 * Sequences: each token carries its position inside its sequence.  A token
 * with position 0 starts a sequence; any other token must directly follow,
 * in the batch, the previous token of its sequence (same adapter, position
 * one lower).  Attention never crosses a sequence boundary.
 *
 * Conventions are those of mlora.h: MLORA_OK / MLORA_E_* return codes,
 * mlora_last_error(), caller-owned device buffers, asynchronous work on the
 * caller's stream, calls on one handle serialised by the caller, device-side
 * range errors reported by mlora_tf_check_status() without trapping (a bad
 * token, target, adapter id or position: the token's logprob is NaN or it
 * is treated as a one-token sequence, and MLORA_E_RANGE is raised).
 * The frozen base and every activation are bf16 (tcgen05 tensor cores, fp32
 * accumulation); the residual stream, norms, softmax statistics, losses and
 * adapter masters are fp32.  Requires an sm_100-family GPU (sm_103a build).
 */
#ifndef MLORA_TF_H
#define MLORA_TF_H

#include "mlora.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct mlora_tf mlora_tf_t;

/* Projection index, in the order of every per-projection array below. */
enum {
    MLORA_TF_Q = 0, MLORA_TF_K = 1, MLORA_TF_V = 2, MLORA_TF_O = 3,
    MLORA_TF_GATE = 4, MLORA_TF_UP = 5, MLORA_TF_DOWN = 6, MLORA_TF_NPROJ = 7
};
#define MLORA_TF_HEAD_DIM 128

typedef struct {
    int32_t vocab;         /* V                                                   */
    int32_t d_model;       /* d, multiple of 128                                  */
    int32_t n_heads;       /* query heads, >= 1                                   */
    int32_t n_kv_heads;    /* key/value heads, divides n_heads                    */
    int32_t head_dim;      /* must be MLORA_TF_HEAD_DIM                           */
    int32_t d_ffn;         /* f, multiple of 128                                  */
    int32_t n_layers;      /* 1 .. 64                                             */
    int32_t n_adapters;    /* 1 .. 1024                                           */
    const int32_t* ranks;  /* host [n_adapters]; 4..MLORA_MAX_RANK, % 4 == 0      */
    const float* alphas;   /* host [n_adapters]                                   */
    float rope_theta;      /* rotary base theta (> 1)                             */
    float rms_eps;         /* RMSNorm epsilon (> 0)                               */
    int64_t max_tokens;    /* largest n_tokens of any call; also the position bound */
} mlora_tf_config;

/* Initial values, read once by mlora_tf_create and copied.  Base tensors are
 * DEVICE pointers to bf16 (raw 16-bit patterns), row-major:
 *   E, Wout [V x d]; final_norm [d];
 *   attn_norm, mlp_norm: HOST arrays [n_layers] of DEVICE pointers to [d];
 *   W[p]: HOST array [n_layers] of DEVICE pointers to W_p [out x in] with
 *     q [n_heads*128 x d], k, v [n_kv_heads*128 x d], o [d x n_heads*128],
 *     gate, up [f x d], down [d x f].
 * Adapters: A[p], B[p] are HOST arrays of n_adapters * n_layers DEVICE
 * pointers to fp32, indexed [a * n_layers + l], with A_p [r x in] and
 * B_p [out x r]; a NULL array or entry initialises that tensor to zero. */
typedef struct {
    const void* E;
    const void* Wout;
    const void* final_norm;
    const void* const* attn_norm;
    const void* const* mlp_norm;
    const void* const* W[MLORA_TF_NPROJ];
    const float* const* A[MLORA_TF_NPROJ];
    const float* const* B[MLORA_TF_NPROJ];
} mlora_tf_init;

/* A flattened token batch: DEVICE int32 arrays of length n_tokens. */
typedef struct {
    int64_t n_tokens;              /* 0 .. max_tokens */
    const int32_t* tokens;
    const int32_t* targets;
    const int32_t* positions;      /* position inside the token's sequence, 0 .. max_tokens-1 */
    const int32_t* adapter_ids;
} mlora_tf_batch;

/* Create a handle (synchronous): validates, allocates all device memory for
 * up to max_tokens tokens, copies and fuses the base (q/k/v stacked, gate/up
 * interleaved, K-major copies for the backward), copies the adapters, zeroes
 * gradients and moments and the step counts.  Errors: E_ARG, E_NOMEM, E_CUDA,
 * E_UNSUPPORTED (no sm_100-family GPU). */
int mlora_tf_create(const mlora_tf_config* cfg, const mlora_tf_init* init, mlora_tf_t** out);
int mlora_tf_destroy(mlora_tf_t* h);

/* Target-token logprobs (no gradient, no state change); logprobs_out DEVICE
 * fp32 [n_tokens]. */
int mlora_tf_forward(mlora_tf_t* h, const mlora_tf_batch* b, float* logprobs_out, void* stream);

/* Forward, loss (mlora_loss kinds of mlora.h, same definitions), adapter-only
 * backward; gradients accumulate until mlora_tf_optim_step.  logprobs_out
 * DEVICE fp32 [n_tokens] and loss_out DEVICE fp64 [n_adapters] may be NULL. */
int mlora_tf_forward_backward(mlora_tf_t* h, const mlora_tf_batch* b, int32_t loss_kind,
                              const mlora_loss_inputs* li, float* logprobs_out, double* loss_out,
                              void* stream);

/* Backpropagate sum_t g_t l_t with the caller's g = dC/dl (DEVICE fp32
 * [n_tokens]) (Deep Dive - Tinker, "The RL datum shape"; the Telegram note on
 * forward_backward_custom). */
int mlora_tf_forward_backward_custom(mlora_tf_t* h, const mlora_tf_batch* b, const float* dloss_dlogprobs,
                                     float* logprobs_out, double* loss_out, void* stream);

/* Per-adapter Adam exactly as mlora_optim_step (same selection, skipping of
 * non-finite gradients, skipped_out). */
int mlora_tf_optim_step(mlora_tf_t* h, const mlora_adam* p, const int32_t* adapters, int32_t n,
                        int32_t* skipped_out, void* stream);

/* Copy one fp32 adapter tensor into dst (DEVICE, caller-owned): projection
 * proj (MLORA_TF_*), factor 0 = A [r x in], 1 = B [out x r]; kind 0 = weight,
 * 1 = accumulated gradient, 2 = first moment, 3 = second moment.  Test and
 * inspection hook. */
int mlora_tf_read_adapter(mlora_tf_t* h, int32_t adapter, int32_t layer, int32_t proj, int32_t factor,
                          int32_t kind, float* dst, void* stream);

/* Step counts: HOST int64 [n_adapters] (synchronises `stream`). */
int mlora_tf_get_steps(mlora_tf_t* h, int64_t* steps_out, void* stream);

/* Synchronise `stream`, return and clear the status word (OK, E_RANGE,
 * E_TIMEOUT). */
int mlora_tf_check_status(mlora_tf_t* h, void* stream);

/* LM-head backward mode, as mlora_set_lm_backward (MLORA_LM_RECOMPUTE, the
 * default of a new handle, or MLORA_LM_KEEP_LOGITS; Tinker API Implementation
 * on TPUs, section 10.4): recompute each row chunk's logits with a second
 * GEMM whose epilogue forms dz, or keep the forward's logits of each chunk as
 * fp16 e = exp(z - m) against each 256-column tile's maximum m (two 16,384 x
 * Vpad fp16 buffers and a second bf16 dz buffer, allocated when selected,
 * freed when left); dz = g (onehot(y) - e exp(m - lse)) in both modes.  Both give bitwise the same results.
 * Synchronises the device.  Errors: E_ARG, E_NOMEM (the handle then stays in
 * the recompute mode), E_CUDA. */
int mlora_tf_set_lm_backward(mlora_tf_t* h, int32_t mode);

/* Attention backward mode (the pages fix only what the backward computes,
 * the gradients of causal attention; this choice of kernels has no
 * counterpart there).  max_seq_len = 0 (the default of a new handle): the
 * query-side kernel recomputes S = Q K^T and dP = dO V^T to form dS and dQ.
 * max_seq_len > 0: the key-side kernel also stores every 128 x 128 block of
 * dS it forms (bf16, the values its dK product reads) and the query side
 * computes dQ = dS K from them, without recomputing; the handle then holds
 * max_tokens-padded/128 x (ceil((S-1)/128) + 1) x n_heads blocks of 32 KB,
 * S = min(max_seq_len, max_tokens), allocated here and freed when the mode
 * is left, and positions must be below S: a token at a larger position is a
 * range error (MLORA_E_RANGE; it is treated as a one-token sequence).  The
 * two modes sum dQ in different orders, so their dQ agree to rounding, not
 * bit for bit; dK and dV are the same.  Synchronises the device.  Errors:
 * E_ARG (max_seq_len < 0, or a layout past 2^31 rows), E_NOMEM (the handle
 * is then in the recompute mode), E_CUDA. */
int mlora_tf_set_attention_backward(mlora_tf_t* h, int32_t max_seq_len);

/* Per-kernel-class timing, as mlora_profile_enable / mlora_profile_read, with
 * the classes below (arrays of MLORA_TF_PROF_CLASSES entries). */
enum {
    MLORA_TF_PROF_ROUTING = 0, MLORA_TF_PROF_EMBED = 1, MLORA_TF_PROF_NORM = 2, MLORA_TF_PROF_SHRINK = 3,
    MLORA_TF_PROF_QKV = 4, MLORA_TF_PROF_ROPE = 5, MLORA_TF_PROF_ATTN_FWD = 6, MLORA_TF_PROF_O = 7,
    MLORA_TF_PROF_GATEUP = 8, MLORA_TF_PROF_DOWN = 9, MLORA_TF_PROF_LM_FWD = 10, MLORA_TF_PROF_LOSS = 11,
    MLORA_TF_PROF_LM_DZ = 12, MLORA_TF_PROF_LM_DH = 13, MLORA_TF_PROF_DOWN_BWD = 14,
    MLORA_TF_PROF_GATEUP_BWD = 15, MLORA_TF_PROF_O_BWD = 16, MLORA_TF_PROF_ATTN_BWD = 17,
    MLORA_TF_PROF_QKV_BWD = 18, MLORA_TF_PROF_GRAD = 19, MLORA_TF_PROF_ADAM = 20, MLORA_TF_PROF_OTHER = 21,
    MLORA_TF_PROF_CLASSES = 22
};
int mlora_tf_profile_enable(mlora_tf_t* h, int32_t on);
int mlora_tf_profile_read(mlora_tf_t* h, double* ms_out, int64_t* launches_out, int32_t reset);

int64_t mlora_tf_kernel_launches(const mlora_tf_t* h);
int64_t mlora_tf_device_bytes(const mlora_tf_t* h);

#ifdef __cplusplus
}
#endif
#endif /* MLORA_TF_H */
