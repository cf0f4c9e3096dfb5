"""Pins of the transformer-block oracle to facts outside itself (CPU only).

Each check ties the fp64 oracle to something it does not compute itself:
central finite differences of the whole step, library routines (torch's
scaled-dot-product attention and rms_norm on the CPU in fp64), closed forms
(one-token sequences attend only to themselves, position 0 is no rotation,
rotation as complex multiplication), invariants the model guarantees
(causality, relative positions, B = 0, adapter isolation, masked targets,
grouped heads equal to repeated heads, loss-kind equivalences), and planted
mistakes that one of these catches.
"""
import numpy as np
import pytest
import torch

import oracle
import oracle.transformer_oracle as to

SHAPE = dict(V=23, d=8, nh=4, nkv=2, hd=4, f=12, L=2)


def tiny_tf(seed=0, ranks=(2, 3, 4), alphas=(4.0, 3.0, 2.0), nkv=None, w_std=0.5, b_std=0.4,
            seq_lens=(5, 1, 7, 4, 6), zero_b=False):
    """A very small fp64 problem with O(1) weights (for finite differences)."""
    s = dict(SHAPE)
    if nkv is not None:
        s["nkv"] = nkv
    V, d, nh, nk, hd, f, L = s["V"], s["d"], s["nh"], s["nkv"], s["hd"], s["f"], s["L"]
    rng = np.random.Generator(np.random.PCG64([99, seed]))
    shapes = to.proj_shapes(d, nh, nk, hd, f)
    base = {"E": rng.standard_normal((V, d)), "Wout": rng.standard_normal((V, d)) * w_std,
            "final_norm": 1 + 0.3 * rng.standard_normal(d),
            "attn_norm": [1 + 0.3 * rng.standard_normal(d) for _ in range(L)],
            "mlp_norm": [1 + 0.3 * rng.standard_normal(d) for _ in range(L)],
            "W": {p: [rng.standard_normal(shapes[p]) * w_std for _ in range(L)] for p in to.PROJ}}
    ad = {"A": {p: [] for p in to.PROJ}, "B": {p: [] for p in to.PROJ}}
    for r in ranks:
        for p in to.PROJ:
            out, inp = shapes[p]
            ad["A"][p].append([rng.standard_normal((r, inp)) * w_std for _ in range(L)])
            ad["B"][p].append([rng.standard_normal((out, r)) * (0.0 if zero_b else b_std)
                               for _ in range(L)])
    n_ad = len(ranks)
    pos, ids = [], []
    for i, T in enumerate(seq_lens):
        pos += list(range(T))
        ids += [int(rng.integers(0, n_ad))] * T
    n = len(pos)
    batch = {"tokens": rng.integers(0, V, n), "targets": rng.integers(0, V, n),
             "positions": np.array(pos), "adapter_ids": np.array(ids),
             "weights": rng.random(n), "advantages": rng.standard_normal(n),
             "noise": rng.standard_normal(n) * 0.3, "dloss": rng.standard_normal(n)}
    o = oracle.TransformerOracle(base, ad, ranks, alphas, s["nh"], s["nkv"], s["hd"],
                                 rope_theta=10.0, rms_eps=1e-6)
    return o, (base, ad, list(ranks), list(alphas), s), batch


def _args(b):
    return b["tokens"], b["targets"], b["positions"], b["adapter_ids"]


def _loss_kw(kind, b, o):
    if kind == "cross_entropy":
        return {"weights": b["weights"]}
    if kind == "custom":
        return {"dloss": b["dloss"]}
    s = o.forward(*_args(b)) + b["noise"]
    return {"advantages": b["advantages"], "sampler_logprobs": s, "clip_eps": 0.2}


def _total_loss(o, b, kind, kw):
    xf, _, groups = o.forward_hidden(b["tokens"], b["positions"], b["adapter_ids"])
    ell, _ = o.logprobs_from_hidden(xf, b["targets"])
    val, _ = oracle.token_loss(kind, ell, **kw)
    return val.sum()


# ------------------------------------------------------ finite differences ---

@pytest.mark.parametrize("kind", ["cross_entropy", "importance_sampling", "ppo", "custom"])
def test_gradients_match_central_differences(kind):
    o, _, b = tiny_tf(seed=1)
    kw = _loss_kw(kind, b, o)
    if kind == "ppo":
        # keep every ratio away from the clip kinks at 1 +- eps
        ell = o.forward(*_args(b))
        r = np.exp(ell - kw["sampler_logprobs"])
        near = np.abs(np.abs(r - 1.0) - 0.2) < 0.02
        kw["advantages"] = np.where(near, 0.0, kw["advantages"])
    o.forward_backward(*_args(b), kind, **kw)
    rng = np.random.Generator(np.random.PCG64([5]))
    h = 1e-5
    worst = 0.0
    for key in o.keys:
        for a in sorted(o.touched):
            for l in range(o.L):
                P = o.P[key][a][l]
                G = o.G[key][a][l]
                for _ in range(3):
                    i = tuple(int(rng.integers(0, s)) for s in P.shape)
                    old = P[i]
                    P[i] = old + h
                    lp = _total_loss(o, b, kind, kw)
                    P[i] = old - h
                    lm = _total_loss(o, b, kind, kw)
                    P[i] = old
                    fd = (lp - lm) / (2 * h)
                    err = abs(fd - G[i]) / max(1e-2, abs(fd))
                    worst = max(worst, err)
                    assert err < 1e-6, (key, a, l, i, fd, G[i])
    assert worst < 1e-6


# ------------------------------------------------------- library routines ---

def test_attention_matches_torch_sdpa():
    rng = np.random.Generator(np.random.PCG64([3]))
    nh, nkv, hd = 6, 2, 8
    lens = [9, 1, 14, 3]
    n = sum(lens)
    q = rng.standard_normal((n, nh * hd)) * 1.5
    k = rng.standard_normal((n, nkv * hd)) * 1.5
    v = rng.standard_normal((n, nkv * hd))
    pos = np.concatenate([np.arange(T) for T in lens])
    seqs = to.sequences(pos, np.zeros(n, int))
    o, lse = to.attention(q, k, v, seqs, nh, nkv, hd)
    for rows in seqs:
        Q = torch.from_numpy(q[rows]).view(len(rows), nh, hd).transpose(0, 1)
        K = torch.from_numpy(k[rows]).view(len(rows), nkv, hd).transpose(0, 1)
        Vv = torch.from_numpy(v[rows]).view(len(rows), nkv, hd).transpose(0, 1)
        K = K.repeat_interleave(nh // nkv, dim=0)
        Vv = Vv.repeat_interleave(nh // nkv, dim=0)
        ref = torch.nn.functional.scaled_dot_product_attention(Q, K, Vv, is_causal=True)
        ref = ref.transpose(0, 1).reshape(len(rows), nh * hd).numpy()
        np.testing.assert_allclose(o[rows], ref, rtol=0, atol=1e-12)
        # lse: log of the normaliser of the same scaled scores
        S = torch.einsum("hqd,hkd->hqk", Q, K) / np.sqrt(hd)
        S = S.masked_fill(~torch.ones(len(rows), len(rows), dtype=torch.bool).tril(), float("-inf"))
        np.testing.assert_allclose(lse[rows], torch.logsumexp(S, -1).T.numpy(), atol=1e-12)


def test_rmsnorm_matches_torch():
    rng = np.random.Generator(np.random.PCG64([4]))
    x = rng.standard_normal((7, 16)) * 3
    g = 1 + rng.standard_normal(16) * 0.2
    y, rstd = to.rmsnorm(x, g, 1e-6)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (16,), torch.from_numpy(g), eps=1e-6)
    np.testing.assert_allclose(y, ref.numpy(), atol=1e-13)
    # its backward against torch autograd of the library routine
    xt = torch.from_numpy(x).requires_grad_(True)
    dy = rng.standard_normal((7, 16))
    torch.nn.functional.rms_norm(xt, (16,), torch.from_numpy(g), eps=1e-6).backward(torch.from_numpy(dy))
    np.testing.assert_allclose(to.rmsnorm_backward(x, g, rstd, dy), xt.grad.numpy(), atol=1e-12)


# ------------------------------------------------------------ closed forms ---

def test_rope_is_complex_rotation_and_identity_at_zero():
    rng = np.random.Generator(np.random.PCG64([6]))
    nh, hd, theta = 3, 8, 10000.0
    x = rng.standard_normal((5, nh * hd))
    pos = np.array([0, 1, 2, 17, 1000])
    y = to.rope(x, pos, nh, hd, theta)
    half = hd // 2
    for hh in range(nh):
        z = x[:, hh * hd: hh * hd + half] + 1j * x[:, hh * hd + half:(hh + 1) * hd]
        w = z * np.exp(1j * pos[:, None] * theta ** (-np.arange(half) / half)[None, :])
        np.testing.assert_allclose(y[:, hh * hd: hh * hd + half], w.real, atol=1e-12)
        np.testing.assert_allclose(y[:, hh * hd + half:(hh + 1) * hd], w.imag, atol=1e-12)
    np.testing.assert_array_equal(y[0], x[0])
    np.testing.assert_allclose(to.rope(y, pos, nh, hd, theta, inverse=True), x, atol=1e-12)


def test_one_token_sequences_attend_to_themselves():
    rng = np.random.Generator(np.random.PCG64([8]))
    nh, nkv, hd = 4, 2, 4
    n = 6
    q, k = rng.standard_normal((n, nh * hd)), rng.standard_normal((n, nkv * hd))
    v = rng.standard_normal((n, nkv * hd))
    seqs = to.sequences(np.zeros(n, int), np.arange(n))
    o, lse = to.attention(q, k, v, seqs, nh, nkv, hd)
    for hq in range(nh):
        hk = hq // (nh // nkv)
        np.testing.assert_array_equal(o[:, hq * hd:(hq + 1) * hd], v[:, hk * hd:(hk + 1) * hd])
        np.testing.assert_allclose(lse[:, hq], (q[:, hq * hd:(hq + 1) * hd] * k[:, hk * hd:(hk + 1) * hd]).sum(1) / 2.0,
                                   atol=1e-14)


# -------------------------------------------------------------- invariants ---

def test_attention_depends_on_relative_positions_only():
    rng = np.random.Generator(np.random.PCG64([9]))
    nh, nkv, hd, theta = 4, 2, 8, 100.0
    lens = [6, 9]
    n = sum(lens)
    pos = np.concatenate([np.arange(T) for T in lens])
    seqs = to.sequences(pos, np.zeros(n, int))
    q, k = rng.standard_normal((n, nh * hd)), rng.standard_normal((n, nkv * hd))
    v = rng.standard_normal((n, nkv * hd))
    o0, _ = to.attention(to.rope(q, pos, nh, hd, theta), to.rope(k, pos, nkv, hd, theta), v, seqs, nh, nkv, hd)
    o1, _ = to.attention(to.rope(q, pos + 37, nh, hd, theta), to.rope(k, pos + 37, nkv, hd, theta), v, seqs,
                         nh, nkv, hd)
    np.testing.assert_allclose(o0, o1, atol=1e-12)
    # but not on absolute ones only: rotating q alone changes the output
    o2, _ = to.attention(to.rope(q, pos + 37, nh, hd, theta), to.rope(k, pos, nkv, hd, theta), v, seqs,
                         nh, nkv, hd)
    assert np.abs(o2 - o0).max() > 1e-3


def test_causal_and_sequence_isolation():
    o, _, b = tiny_tf(seed=2)
    lp = o.forward(*_args(b))
    b2 = {k: np.array(v, copy=True) for k, v in b.items()}
    # change the last two inputs of the third sequence (tokens 6..12)
    b2["tokens"][11:13] = (b2["tokens"][11:13] + 5) % SHAPE["V"]
    lp2 = o.forward(*_args(b2))
    changed = np.nonzero(lp2 != lp)[0]
    assert set(changed.tolist()) <= {11, 12} and 12 in changed.tolist()


def test_zero_b_reproduces_base():
    o, (base, ad, ranks, alphas, s), b = tiny_tf(seed=3, zero_b=True)
    lp = o.forward(*_args(b))
    for p in to.PROJ:
        for a in range(len(ranks)):
            for l in range(s["L"]):
                o.P["A_" + p][a][l] = np.zeros_like(o.P["A_" + p][a][l])
    np.testing.assert_array_equal(o.forward(*_args(b)), lp)


def test_mixed_batch_equals_separate_adapter_runs():
    o, parts, b = tiny_tf(seed=4)
    kw = {"weights": b["weights"]}
    res = o.forward_backward(*_args(b), "cross_entropy", **kw)
    ids = b["adapter_ids"]
    for a in sorted(set(ids.tolist())):
        oa, _, _ = tiny_tf(seed=4)
        rows = np.nonzero(ids == a)[0]
        sub = {k: (v[rows] if isinstance(v, np.ndarray) and v.shape[:1] == ids.shape else v) for k, v in b.items()}
        ra = oa.forward_backward(*_args(sub), "cross_entropy", weights=sub["weights"])
        np.testing.assert_allclose(ra["logprobs"], res["logprobs"][rows], atol=1e-12)
        for key in o.keys:
            for l in range(o.L):
                np.testing.assert_allclose(oa.G[key][a][l], o.G[key][a][l], atol=1e-11, rtol=1e-10)
                for other in range(o.n_adapters):
                    if other != a:
                        assert not oa.G[key][other][l].any()


def test_masked_targets_contribute_nothing():
    o, _, b = tiny_tf(seed=5)
    w = b["weights"].copy()
    w[::3] = 0.0
    o.forward_backward(*_args(b), "cross_entropy", weights=w)
    o2, _, _ = tiny_tf(seed=5)
    b2 = dict(b)
    b2["targets"] = b["targets"].copy()
    b2["targets"][::3] = (b2["targets"][::3] + 7) % SHAPE["V"]
    o2.forward_backward(*_args(b2), "cross_entropy", weights=w)
    for key in o.keys:
        for a in range(o.n_adapters):
            for l in range(o.L):
                np.testing.assert_allclose(o2.G[key][a][l], o.G[key][a][l], atol=1e-12)


def test_grouped_heads_equal_repeated_heads():
    o, (base, ad, ranks, alphas, s), b = tiny_tf(seed=6)
    lp = o.forward(*_args(b))
    grp, hd = s["nh"] // s["nkv"], s["hd"]

    def rep_rows(w):   # [nkv*hd x ...] -> [nh*hd x ...], head j <- head j // grp
        return np.concatenate([w[(j // grp) * hd:(j // grp + 1) * hd] for j in range(s["nh"])])

    base2 = dict(base)
    base2["W"] = dict(base["W"])
    ad2 = {"A": dict(ad["A"]), "B": dict(ad["B"])}
    for p in ("k", "v"):
        base2["W"][p] = [rep_rows(w) for w in base["W"][p]]
        ad2["B"][p] = [[rep_rows(w) for w in row] for row in ad["B"][p]]
    o2 = oracle.TransformerOracle(base2, ad2, ranks, alphas, s["nh"], s["nh"], hd, rope_theta=10.0)
    np.testing.assert_allclose(o2.forward(*_args(b)), lp, atol=1e-12)


def test_loss_kind_equivalences():
    o1, _, b = tiny_tf(seed=7)
    o2, _, _ = tiny_tf(seed=7)
    o1.forward_backward(*_args(b), "cross_entropy", weights=b["weights"])
    o2.forward_backward_custom(*_args(b), -b["weights"])
    o3, _, _ = tiny_tf(seed=7)
    ell = o3.forward(*_args(b))
    o3.forward_backward(*_args(b), "importance_sampling", advantages=b["weights"], sampler_logprobs=ell)
    for key in o1.keys:
        for a in range(o1.n_adapters):
            for l in range(o1.L):
                np.testing.assert_array_equal(o2.G[key][a][l], o1.G[key][a][l])
                np.testing.assert_allclose(o3.G[key][a][l], o1.G[key][a][l], atol=1e-12, rtol=1e-10)


def test_sequences_reject_broken_layout():
    with pytest.raises(ValueError):
        to.sequences([0, 1, 3], [0, 0, 0])
    with pytest.raises(ValueError):
        to.sequences([0, 1, 2], [0, 0, 1])
    with pytest.raises(ValueError):
        to.sequences([1, 2], [0, 0])
    assert [s.tolist() for s in to.sequences([0, 1, 0, 0, 1], [0, 0, 1, 0, 0])] == [[0, 1], [2], [3, 4]]


# ------------------------------------------------------ planted mistakes ---

def _fd_fails(monkeypatch, name, bad):
    monkeypatch.setattr(to, name, bad)
    with pytest.raises(AssertionError):
        test_gradients_match_central_differences("cross_entropy")


def test_planted_rope_backward_sign_is_caught(monkeypatch):
    good = to.rope
    _fd_fails(monkeypatch, "rope",
              lambda x, pos, nh, hd, th, inverse=False: good(x, pos, nh, hd, th, inverse=False))


def test_planted_rmsnorm_backward_is_caught(monkeypatch):
    _fd_fails(monkeypatch, "rmsnorm_backward",
              lambda x, g, rstd, dy: rstd[:, None] * dy * g[None, :])


def test_planted_attention_dk_transpose_is_caught(monkeypatch):
    good = to.attention_backward

    def bad(q, k, v, do, seqs, nh, nkv, hd):
        dq, dk, dv = good(q, k, v, do, seqs, nh, nkv, hd)
        return dq, dk * 0.5, dv
    _fd_fails(monkeypatch, "attention_backward", bad)


def test_planted_head_grouping_is_caught(monkeypatch):
    def bad(q, k, v, seqs, nh, nkv, hd):     # query head j reads kv head j % nkv
        qq = q.copy()
        grp = nh // nkv
        order = [(j % nkv) * grp + j // nkv for j in range(nh)]
        for j in range(nh):
            qq[:, order[j] * hd:(order[j] + 1) * hd] = q[:, j * hd:(j + 1) * hd]
        o, lse = good(qq, k, v, seqs, nh, nkv, hd)
        out = o.copy()
        for j in range(nh):
            out[:, j * hd:(j + 1) * hd] = o[:, order[j] * hd:(order[j] + 1) * hd]
        return out, lse
    good = to.attention
    monkeypatch.setattr(to, "attention", bad)
    with pytest.raises(AssertionError):
        test_grouped_heads_equal_repeated_heads()
