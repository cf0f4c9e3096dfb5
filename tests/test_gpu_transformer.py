"""GPU parity of the transformer-block step (RMSNorm, grouped-head causal
attention with rotary positions, gated SiLU MLP, LoRA on all seven
projections) through the C ABI, against the CPU oracle.

Tolerances.  Logprobs: max abs error <= 2e-2 and post-Adam adapter weights:
relative Frobenius error <= 1e-2 per (adapter, layer, tensor) -- the
specification's bounds for a bf16 base with fp32 accumulation.  Adapter
gradients: a bound derived for this block.  Its activations are stored in
bf16 between kernels (the normalised inputs of the projections, q, k, v, the
attention output, the gate/up values, the backward's dh, dO and dS), and
that storage by itself -- the fp64 definition evaluated with only those
values rounded to bf16 -- moves the exact gradients by up to 1.1 % (median
0.65 %) on the workloads' N(0, 0.02) weights and by up to 1.7 % when q / k
are drawn at 0.08 so that the attention scores spread as at the 8B widths
(query entries of standard deviation ~1.3).  The GPU is an independent
rounding of the same size, so gradients are checked at <= 2.5e-2 per tensor
and a median over all tensors <= 1.5e-2.

Inputs are seeded; the sampler logprobs of IS / PPO come from an oracle
forward, and PPO tokens whose ratio lies within 3 % of a clip kink get a zero
advantage on both sides (there the branch is decided by rounding).  Sizes span
several 128-row tiles, sequences that cross tiles, several sequences per tile,
and ragged segment tails.
"""
import numpy as np
import pytest

import oracle
import workloads.transformer as wt
from _gpu_util import dev, rel_fro

pytestmark = pytest.mark.gpu

LP_TOL = 2e-2
W_TOL = 1e-2           # post-Adam weights
GRAD_TOL = 2.5e-2      # gradients, per tensor
GRAD_MEDIAN_TOL = 1.5e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def _make(cfg, base, ad, max_tokens, lm=None, attn=0):
    import rl_step_gb300.transformer as t
    dbase = {"E": dev(base["E"]), "Wout": dev(base["Wout"]), "final_norm": dev(base["final_norm"]),
             "attn_norm": [dev(g) for g in base["attn_norm"]], "mlp_norm": [dev(g) for g in base["mlp_norm"]],
             "W": {p: [dev(w) for w in base["W"][p]] for p in t.PROJ}}
    A = {p: [[dev(x) for x in row] for row in ad["A"][p]] for p in t.PROJ}
    B = {p: [[dev(x) for x in row] for row in ad["B"][p]] for p in t.PROJ}
    h = t.tf_create(cfg.vocab, cfg.d_model, cfg.n_heads, cfg.n_kv_heads, cfg.d_ffn, cfg.n_layers,
                    cfg.ranks, cfg.alphas, max_tokens, dbase, A, B, rope_theta=cfg.rope_theta,
                    rms_eps=cfg.rms_eps)
    if lm is not None:
        t.tf_set_lm_backward(h, lm)
    if attn:
        t.tf_set_attention_backward(h, attn)
    return h


def _oracle(cfg, base, ad):
    return oracle.TransformerOracle(base, ad, cfg.ranks, cfg.alphas, cfg.n_heads, cfg.n_kv_heads,
                                    cfg.head_dim, cfg.rope_theta, cfg.rms_eps)


def _args(b):
    return b["tokens"], b["targets"], b["positions"], b["adapter_ids"]


def _dargs(b):
    return tuple(dev(x) for x in _args(b))


def _problem(**overrides):
    cfg = wt.get_tf_config("tf_small", **overrides)
    base = wt.make_tf_base_weights(cfg)
    ad = wt.make_tf_adapters(cfg)
    b = wt.make_tf_batch(cfg)
    lp0 = _oracle(cfg, base, ad).forward(*_args(b))
    # PPO: no token within 3 % of a clip kink (the branch there is a rounding decision)
    r = np.exp(-b["sampler_noise"].astype(np.float64))
    near = (np.abs(r - (1 + b["clip_eps"])) < 0.03) | (np.abs(r - (1 - b["clip_eps"])) < 0.03)
    b["advantages"] = np.where(near, 0.0, b["advantages"]).astype(np.float32)
    return cfg, base, ad, b, lp0


@pytest.fixture(scope="module")
def small():
    return _problem()


@pytest.fixture(scope="module")
def sharp():
    return _problem(qk_std=0.08)


def _gpu_step(h, b, kind, s):
    import rl_step_gb300.transformer as t
    if kind == "custom":
        return t.tf_forward_backward_custom(h, *_dargs(b), dev(b["dloss"]))
    if kind == "cross_entropy":
        return t.tf_forward_backward(h, *_dargs(b), kind, weights=dev(b["weights"]))
    return t.tf_forward_backward(h, *_dargs(b), kind, advantages=dev(b["advantages"]),
                                 sampler_logprobs=dev(s.astype(np.float32)), clip_eps=b["clip_eps"])


def _oracle_step(o, b, kind, s):
    if kind == "custom":
        return o.forward_backward_custom(*_args(b), b["dloss"])
    if kind == "cross_entropy":
        return o.forward_backward(*_args(b), kind, weights=b["weights"])
    return o.forward_backward(*_args(b), kind, advantages=b["advantages"], sampler_logprobs=s,
                              clip_eps=b["clip_eps"])


def _tensor_errors(h, o, adapters, kind):
    """(max, (adapter, layer, proj, factor) of the max, median) relative
    Frobenius error over the adapters' tensors."""
    import rl_step_gb300.transformer as t
    worst, where, all_e = 0.0, None, []
    for a in adapters:
        for l in range(o.L):
            for p in t.PROJ:
                for fac in ("A", "B"):
                    x = t.tf_read_adapter(h, a, l, p, fac, kind).cpu().numpy()
                    ref = (o.G if kind == "grad" else o.P)[f"{fac}_{p}"][a][l]
                    e = rel_fro(x, ref)
                    all_e.append(e)
                    if e > worst:
                        worst, where = e, (a, l, p, fac)
    return worst, where, float(np.median(all_e))


def _check_grads(h, o, adapters):
    err, where, med = _tensor_errors(h, o, adapters, "grad")
    assert err <= GRAD_TOL and med <= GRAD_MEDIAN_TOL, (err, where, med)


def test_forward_matches_oracle(small):
    import rl_step_gb300.transformer as t
    cfg, base, ad, b, lp0 = small
    h = _make(cfg, base, ad, len(b["tokens"]))
    lp = t.tf_forward(h, *_dargs(b)).cpu().numpy()
    assert t.tf_check_status(h) == 0
    err = float(np.max(np.abs(lp - lp0)))
    assert np.isfinite(lp).all() and err <= LP_TOL, err


def _step_and_adam(prob, kind, lm=None, attn=0):
    import rl_step_gb300.transformer as t
    cfg, base, ad, b, lp0 = prob
    s = lp0 + b["sampler_noise"]
    h = _make(cfg, base, ad, len(b["tokens"]), lm, attn)
    o = _oracle(cfg, base, ad)
    lp, loss = _gpu_step(h, b, kind, s)
    ref = _oracle_step(o, b, kind, s)
    assert t.tf_check_status(h) == 0
    assert float(np.max(np.abs(lp.cpu().numpy() - ref["logprobs"]))) <= LP_TOL
    scale = np.array([np.abs(ref["loss_per_adapter"][a]) for a in range(cfg.n_adapters)]).sum() + 1.0
    assert float(np.max(np.abs(loss.cpu().numpy() - ref["loss_per_adapter"]))) <= 2e-2 * scale
    touched = sorted(set(b["adapter_ids"].tolist()))
    _check_grads(h, o, touched)
    t.tf_optim_step(h, lr=cfg.lr)
    o.optim_step(lr=cfg.lr)
    assert t.tf_check_status(h) == 0
    err, where, _ = _tensor_errors(h, o, touched, "weight")
    assert err <= W_TOL, (err, where)
    assert t.tf_get_steps(h) == o.step


@pytest.mark.parametrize("lm", ["recompute", "keep_logits"])
@pytest.mark.parametrize("kind", ["ppo", "cross_entropy", "importance_sampling", "custom"])
def test_step_and_adam_match_oracle(small, kind, lm):
    _step_and_adam(small, kind, lm)


def test_lm_backward_modes_agree_over_three_chunks():
    """Recomputing each LM-head chunk's logits and keeping them give bitwise
    the same logprobs and losses, and the same gradients up to the arrival
    order of the fp32 gradient atomics, on a batch of three LM-head chunks; the
    kept-logits mode holds two chunks of fp16 e = exp(z - tile max) and a
    second dz chunk more."""
    import rl_step_gb300.transformer as t
    cfg = wt.get_tf_config("tf_small")
    base, ad = wt.make_tf_base_weights(cfg), wt.make_tf_adapters(cfg)
    b = wt.make_tf_batch(cfg, 40000)
    N = len(b["tokens"])
    res = {}
    for lm in ("keep_logits", "recompute"):
        h = _make(cfg, base, ad, N, lm)
        lp, loss = t.tf_forward_backward(h, *_dargs(b), "cross_entropy", weights=dev(b["weights"]))
        assert t.tf_check_status(h) == 0
        g = {(a, l, p, fac): t.tf_read_adapter(h, a, l, p, fac, "grad").cpu().numpy()
             for a in range(cfg.n_adapters) for l in range(cfg.n_layers) for p in t.PROJ for fac in ("A", "B")}
        res[lm] = (lp.cpu().numpy(), loss.cpu().numpy(), g, h.device_bytes)
        del h
    (lp_k, loss_k, g_k, by_k), (lp_r, loss_r, g_r, by_r) = res["keep_logits"], res["recompute"]
    assert np.array_equal(lp_k, lp_r) and np.array_equal(loss_k, loss_r)
    assert max(rel_fro(g_r[k], g_k[k]) for k in g_k) <= 1e-4
    tiles = -(-(N + 127 * min(N, cfg.n_adapters)) // 128)
    assert tiles > 256
    vpad = (cfg.vocab + 63) // 64 * 64
    assert by_k - by_r == 128 * 128 * vpad * (2 + 2 * 2)          # a dz chunk, two fp16 e chunks


@pytest.mark.parametrize("kind", ["ppo", "custom"])
def test_sharp_attention_step_matches_oracle(sharp, kind):
    _step_and_adam(sharp, kind)


# The stored-dS attention backward: the key side stores every dS block and the
# query side forms dQ = dS K from them.  tf_small's sequences are at most 300
# tokens long (a query tile then sees at most four key tiles).
SEQ_HI_SMALL = 300


@pytest.mark.parametrize("prob", ["small", "sharp"])
@pytest.mark.parametrize("kind", ["ppo", "cross_entropy", "custom"])
def test_stored_ds_step_matches_oracle(request, prob, kind):
    _step_and_adam(request.getfixturevalue(prob), kind, attn=SEQ_HI_SMALL)


def test_attention_backward_modes_agree_and_bound_positions(small):
    """Both attention backward modes give the same logprobs and losses bit for
    bit (the forward is shared) and gradients equal to rounding (dQ is summed in
    another order); the stored mode holds max_tiles x ktc x n_heads blocks of
    32 KB more, and a position past its sequence bound is a range error."""
    import rl_step_gb300.transformer as t
    cfg, base, ad, b, _ = small
    N = len(b["tokens"])
    res = {}
    for attn in (0, SEQ_HI_SMALL):
        h = _make(cfg, base, ad, N, attn=attn)
        lp, loss = t.tf_forward_backward(h, *_dargs(b), "cross_entropy", weights=dev(b["weights"]))
        assert t.tf_check_status(h) == 0
        g = {(a, l, p, fac): t.tf_read_adapter(h, a, l, p, fac, "grad").cpu().numpy()
             for a in range(cfg.n_adapters) for l in range(cfg.n_layers) for p in t.PROJ for fac in ("A", "B")}
        res[attn] = (lp.cpu().numpy(), loss.cpu().numpy(), g, h.device_bytes)
        if attn:
            long_seq = _layout(cfg, [SEQ_HI_SMALL + 5, 3], [0, 1], 11)
            t.tf_forward_backward(h, *_dargs(long_seq), "cross_entropy", weights=dev(long_seq["weights"]))
            assert t.tf_check_status(h) == -2
            assert t.tf_check_status(h) == 0
            stored_bytes = h.device_bytes
            import rl_step_gb300 as m
            with pytest.raises(m.MLoRAError):
                t.tf_set_attention_backward(h, -1)
            assert h.device_bytes == stored_bytes           # a rejected call changes nothing
            t.tf_set_attention_backward(h, 0)               # back to recomputing: the blocks are freed
            res["left"] = h.device_bytes
            t.tf_forward_backward(h, *_dargs(long_seq), "cross_entropy", weights=dev(long_seq["weights"]))
            assert t.tf_check_status(h) == 0                # positions are bounded by max_tokens again
        del h
    (lp_r, loss_r, g_r, by_r), (lp_s, loss_s, g_s, by_s) = res[0], res[SEQ_HI_SMALL]
    assert np.array_equal(lp_r, lp_s) and np.array_equal(loss_r, loss_s)
    assert max(rel_fro(g_s[k], g_r[k]) for k in g_r) <= 1e-2
    max_tiles = -(-(N + 127 * min(N, cfg.n_adapters)) // 128)
    ktc = -(-(SEQ_HI_SMALL - 1) // 128) + 1
    assert by_s - by_r == max_tiles * ktc * cfg.n_heads * 128 * 128 * 2
    assert res["left"] == by_r


def test_sharp_attention_forward_matches_oracle(sharp):
    import rl_step_gb300.transformer as t
    cfg, base, ad, b, lp0 = sharp
    h = _make(cfg, base, ad, len(b["tokens"]))
    lp = t.tf_forward(h, *_dargs(b)).cpu().numpy()
    assert t.tf_check_status(h) == 0
    assert float(np.max(np.abs(lp - lp0))) <= LP_TOL


def test_gradients_accumulate_across_calls(small):
    import rl_step_gb300.transformer as t
    cfg, base, ad, b, lp0 = small
    h = _make(cfg, base, ad, len(b["tokens"]))
    o = _oracle(cfg, base, ad)
    for _ in range(2):
        _gpu_step(h, b, "cross_entropy", None)
        _oracle_step(o, b, "cross_entropy", None)
    _check_grads(h, o, sorted(set(b["adapter_ids"].tolist())))


def _layout(cfg, lens, ads, seed):
    rng = np.random.Generator(np.random.PCG64([seed]))
    n = sum(lens)
    return {"tokens": rng.integers(0, cfg.vocab, n).astype(np.int32),
            "targets": rng.integers(0, cfg.vocab, n).astype(np.int32),
            "positions": np.concatenate([np.arange(T) for T in lens]).astype(np.int32),
            "adapter_ids": np.concatenate([np.full(T, a) for T, a in zip(lens, ads)]).astype(np.int32),
            "weights": (rng.random(n) < 0.7).astype(np.float32),
            "dloss": rng.standard_normal(n).astype(np.float32)}


@pytest.mark.parametrize("lens,ads", [
    ([1, 1, 1, 1, 1], [0, 1, 2, 0, 1]),                       # one-token sequences
    ([300], [1]),                                              # one sequence over three tiles
    ([1], [2]),                                                # a single token
    ([129, 127, 1, 255, 2, 130], [0, 0, 0, 2, 2, 1]),          # ragged tiles, several per tile
])
@pytest.mark.parametrize("attn", [0, SEQ_HI_SMALL])
def test_edge_layouts_match_oracle(small, lens, ads, attn):
    import rl_step_gb300.transformer as t
    cfg, base, ad, _, _ = small
    b = _layout(cfg, lens, ads, sum(lens))
    h = _make(cfg, base, ad, 1024, attn=attn)
    o = _oracle(cfg, base, ad)
    lp, _ = _gpu_step(h, b, "cross_entropy", None)
    ref = _oracle_step(o, b, "cross_entropy", None)
    assert t.tf_check_status(h) == 0
    assert float(np.max(np.abs(lp.cpu().numpy() - ref["logprobs"]))) <= LP_TOL
    _check_grads(h, o, sorted(set(ads)))


def test_custom_with_minus_weights_equals_cross_entropy(small):
    import rl_step_gb300.transformer as t
    cfg, base, ad, b, _ = small
    h1 = _make(cfg, base, ad, len(b["tokens"]))
    h2 = _make(cfg, base, ad, len(b["tokens"]))
    t.tf_forward_backward(h1, *_dargs(b), "cross_entropy", weights=dev(b["weights"]))
    t.tf_forward_backward_custom(h2, *_dargs(b), dev(-b["weights"]))
    for a in sorted(set(b["adapter_ids"].tolist())):
        for p in t.PROJ:
            for fac in ("A", "B"):
                x1 = t.tf_read_adapter(h1, a, 1, p, fac, "grad").cpu().numpy()
                x2 = t.tf_read_adapter(h2, a, 1, p, fac, "grad").cpu().numpy()
                assert rel_fro(x2, x1) <= 1e-5


def test_empty_batch_and_bad_positions(small):
    import torch
    import rl_step_gb300.transformer as t
    cfg, base, ad, b, _ = small
    h = _make(cfg, base, ad, 256)
    e = torch.empty(0, dtype=torch.int32, device="cuda")
    lp, loss = t.tf_forward_backward(h, e, e, e, e, "cross_entropy", weights=torch.empty(0, device="cuda"))
    assert loss.cpu().numpy().tolist() == [0.0] * cfg.n_adapters
    bad = _layout(cfg, [4, 3], [0, 1], 5)
    bad["positions"][5] = 7                   # breaks its sequence
    lp = t.tf_forward(h, *_dargs(bad)).cpu().numpy()
    assert t.tf_check_status(h) == -2
    assert np.isfinite(lp).all()
    assert t.tf_check_status(h) == 0
