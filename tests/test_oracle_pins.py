"""Pins of the CPU oracle to facts outside itself (CPU only).

Each test checks the oracle against something the pages or the mathematics
fix: a pure-Python brute force of the definitions, closed forms (Wout = 0,
Adam at t = 1, PPO at the clip boundaries), central finite differences,
library routines (scipy's log_softmax), invariants the method guarantees
(B = 0 reproduces the base, adapter isolation, masked tokens, loss-kind
equivalences) and the pages' worked examples.  The last tests plant mistakes
in the oracle and check that a pin catches each one.
"""
import math

import numpy as np
import pytest
import scipy.special

import oracle
import oracle.mlora_oracle as om
from _util import golden, tiny_problem


def _make(seed_shift=0, **kw):
    base, ad, ranks, alphas, batch = tiny_problem(seed_shift, **kw)
    return oracle.Oracle(base, ad, ranks, alphas), (base, ad, ranks, alphas), batch


# ---------------------------------------------------------------- routing ---

def _routing_brute(ids, n_ad, tile):
    perm = []
    for a in range(n_ad):
        for t, x in enumerate(ids):
            if x == a:
                perm.append(t)
    counts = [sum(1 for x in ids if x == a) for a in range(n_ad)]
    seg, pad, tiles = [0], [0], []
    for a in range(n_ad):
        seg.append(seg[-1] + counts[a])
        nt = -(-counts[a] // tile)
        pad.append(pad[-1] + nt * tile)
        tiles += [a] * nt
    return perm, seg, pad, tiles


@pytest.mark.parametrize("n,n_ad,tile", [(1, 1, 128), (7, 3, 4), (300, 5, 128),
                                         (1000, 17, 128), (64, 8, 8), (0, 4, 128)])
def test_routing_matches_brute_force(n, n_ad, tile):
    rng = np.random.Generator(np.random.PCG64([11, n, n_ad]))
    ids = rng.integers(0, n_ad, n)
    if n > 10:
        ids[ids == (n_ad - 1)] = 0   # leave one adapter empty
    r = oracle.routing(ids, n_ad, tile)
    perm, seg, pad, tiles = _routing_brute(list(ids), n_ad, tile)
    assert r["perm"].tolist() == perm
    assert r["seg_off"].tolist() == seg
    assert r["pad_off"].tolist() == pad
    assert r["tile_ad"].tolist() == tiles
    # permutation, stable, contiguous segments
    assert sorted(r["perm"].tolist()) == list(range(n))
    for a in range(n_ad):
        seg_rows = r["perm"][r["seg_off"][a]:r["seg_off"][a + 1]]
        assert (ids[seg_rows] == a).all()
        assert (np.diff(seg_rows) > 0).all()


def test_routing_rejects_out_of_range():
    with pytest.raises(ValueError):
        oracle.routing([0, 3], 3)


# ---------------------------------------------------------------- forward ---

def _brute_logprob(params, tok, tgt, a, use_lora=True):
    """Pure-Python evaluation of the definitions for one token."""
    base, ad, ranks, alphas = params
    E = base["E"].astype(float).tolist()
    h = list(E[tok])
    L = len(base["W1"])
    gam = alphas[a] / ranks[a]

    def mv(M, x):
        return [math.fsum(mi * xi for mi, xi in zip(row, x)) for row in M]

    for l in range(L):
        W1 = base["W1"][l].astype(float).tolist()
        W2 = base["W2"][l].astype(float).tolist()
        u = mv(W1, h)
        if use_lora:
            v1 = mv(ad["A1"][a][l].astype(float).tolist(), h)
            ex = mv(ad["B1"][a][l].astype(float).tolist(), v1)
            u = [ui + gam * e for ui, e in zip(u, ex)]
        act = [ui / (1.0 + math.exp(-ui)) for ui in u]
        y = mv(W2, act)
        if use_lora:
            v2 = mv(ad["A2"][a][l].astype(float).tolist(), act)
            ex = mv(ad["B2"][a][l].astype(float).tolist(), v2)
            y = [yi + gam * e for yi, e in zip(y, ex)]
        h = [hi + yi for hi, yi in zip(h, y)]
    z = mv(base["Wout"].astype(float).tolist(), h)
    lse = math.log(math.fsum(math.exp(zv) for zv in z))
    return z[tgt] - lse


def test_forward_matches_pure_python():
    o, params, b = _make(1)
    ell = o.forward(b["tokens"], b["targets"], b["adapter_ids"])
    for t in range(6):
        ref = _brute_logprob(params, int(b["tokens"][t]), int(b["targets"][t]),
                             int(b["adapter_ids"][t]))
        assert abs(ell[t] - ref) < 1e-12 * max(1.0, abs(ref))


def test_forward_wout_zero_gives_minus_log_v():
    o, params, b = _make(2)
    o.Wout[...] = 0.0
    ell = o.forward(b["tokens"], b["targets"], b["adapter_ids"])
    assert np.all(ell == -np.log(o.V))


def test_b_zero_reproduces_base():
    o, params, b = _make(3)
    for k in ("B1", "B2"):
        for a in range(o.n_adapters):
            for l in range(o.L):
                o.P[k][a][l][...] = 0.0
    ell = o.forward(b["tokens"], b["targets"], b["adapter_ids"])
    base = params[0]
    h = base["E"].astype(np.float64)[b["tokens"]]
    for l in range(o.L):
        u = h @ base["W1"][l].astype(np.float64).T
        h = h + (u / (1 + np.exp(-u))) @ base["W2"][l].astype(np.float64).T
    z = h @ base["Wout"].astype(np.float64).T
    ref = scipy.special.log_softmax(z, axis=1)[np.arange(len(h)), b["targets"]]
    assert np.array_equal(ell, ell)  # finite
    np.testing.assert_allclose(ell, ref, rtol=0, atol=1e-12)
    for t in range(3):
        bp = _brute_logprob(params, int(b["tokens"][t]), int(b["targets"][t]), 0,
                            use_lora=False)
        assert abs(ell[t] - bp) < 1e-12 * max(1.0, abs(bp))


def test_logsumexp_matches_scipy_and_identity():
    rng = np.random.Generator(np.random.PCG64([5]))
    z = rng.standard_normal((9, 33)) * 30.0
    lse = oracle.logsumexp_rows(z)
    np.testing.assert_allclose(lse, scipy.special.logsumexp(z, axis=1), rtol=1e-15, atol=0)
    np.testing.assert_allclose(np.log(np.exp(z - lse[:, None]).sum(axis=1)), 0.0, atol=1e-14)


# ---------------------------------------------------------------- losses ----

def test_ppo_boundaries_closed_form():
    g = golden("ppo_boundaries.json")
    for row in g["rows"]:
        ell = np.array([math.log(row["r"])])
        r = float(np.exp(ell[0]))
        eps = g["eps"]
        if row.get("tie") == "upper":
            eps = r - 1.0
        elif row.get("tie") == "lower":
            eps = 1.0 - r
        val, dl = oracle.token_loss("ppo", ell, advantages=np.array([row["A"]]),
                                    sampler_logprobs=np.zeros(1), clip_eps=eps)
        assert abs(val[0] - row["value"]) < 1e-12, row
        assert abs(dl[0] - row["dl"]) < 1e-12, row


def test_nonfinite_inputs_are_contained():
    ell = np.array([-1.0, -2.0, np.nan, -1.0, -1.0])
    A = np.array([1.0, np.inf, 1.0, 1.0, 1.0])
    s = np.array([0.0, 0.0, 0.0, np.nan, -1000.0])      # last: ratio overflows
    for kind in ("importance_sampling", "ppo"):
        val, g = oracle.token_loss(kind, ell, advantages=A, sampler_logprobs=s)
        assert np.isfinite(val).all() and np.isfinite(g).all()
        assert (g[1:] == 0).all() and (val[1:] == 0).all()
        assert g[0] != 0
    w = np.array([1.0, np.nan, 1.0, 0.0, 1.0])
    val, g = oracle.token_loss("cross_entropy", ell, weights=w)
    assert g.tolist() == [-1.0, 0.0, 0.0, 0.0, -1.0]


# ---------------------------------------------------------------- gradients -

def _fd_check(kind, seed_shift=4, n_per=2, h=1e-5):
    """Max relative error between oracle grads and central differences."""
    o, params, b = _make(seed_shift)
    ids = b["adapter_ids"]
    ell0 = o.forward(b["tokens"], b["targets"], ids)
    s = ell0 + b["noise"]
    kw = dict(weights=b["weights"], advantages=b["advantages"], sampler_logprobs=s,
              clip_eps=0.2, dloss=b["dloss"])
    if kind == "ppo":
        r = np.exp(ell0 - s)
        assert np.min(np.abs(np.abs(r - 1.0) - 0.2)) > 1e-3   # away from the kinks
    o.forward_backward(b["tokens"], b["targets"], ids, kind, **kw)

    def loss_of(oo):
        ell = oo.forward(b["tokens"], b["targets"], ids)
        return math.fsum(oracle.token_loss(kind, ell, **kw)[0])

    rng = np.random.Generator(np.random.PCG64([99, seed_shift]))
    num, ana = [], []
    for k in oracle.TENSORS:
        for a in range(o.n_adapters):
            for l in range(o.L):
                P = o.P[k][a][l]
                for _ in range(n_per):
                    i = tuple(int(rng.integers(0, n)) for n in P.shape)
                    x0 = P[i]
                    P[i] = x0 + h
                    lp = loss_of(o)
                    P[i] = x0 - h
                    lm = loss_of(o)
                    P[i] = x0
                    num.append((lp - lm) / (2 * h))
                    ana.append(o.G[k][a][l][i])
    num, ana = np.array(num), np.array(ana)
    return np.linalg.norm(num - ana) / np.linalg.norm(ana)


@pytest.mark.parametrize("kind", ["cross_entropy", "importance_sampling", "ppo", "custom"])
def test_gradients_match_finite_differences(kind):
    assert _fd_check(kind) < 1e-6


def test_mixed_batch_equals_separate_runs():
    o, params, b = _make(5)
    kw = dict(weights=b["weights"])
    out = o.forward_backward(b["tokens"], b["targets"], b["adapter_ids"], "cross_entropy", **kw)
    for a in range(o.n_adapters):
        rows = np.nonzero(b["adapter_ids"] == a)[0]
        o2 = oracle.Oracle(*[params[0], params[1], params[2], params[3]])
        out2 = o2.forward_backward(b["tokens"][rows], b["targets"][rows], b["adapter_ids"][rows],
                                   "cross_entropy", weights=b["weights"][rows])
        np.testing.assert_allclose(out["logprobs"][rows], out2["logprobs"], rtol=1e-13, atol=0)
        assert abs(out["loss_per_adapter"][a] - out2["loss_per_adapter"][a]) < 1e-12
        for k in oracle.TENSORS:
            for l in range(o.L):
                np.testing.assert_allclose(o.G[k][a][l], o2.G[k][a][l], rtol=1e-11, atol=1e-15)
                for a2 in range(o.n_adapters):
                    if a2 != a:
                        assert not o2.G[k][a2][l].any()   # no leak into other adapters


def test_masked_tokens_contribute_nothing():
    o, params, b = _make(6)
    w = b["weights"].copy()
    w[::3] = 0.0
    o.forward_backward(b["tokens"], b["targets"], b["adapter_ids"], "cross_entropy", weights=w)
    tok2, tgt2 = b["tokens"].copy(), b["targets"].copy()
    tok2[::3] = (tok2[::3] + 5) % o.V
    tgt2[::3] = (tgt2[::3] + 7) % o.V
    o2 = oracle.Oracle(*params)
    o2.forward_backward(tok2, tgt2, b["adapter_ids"], "cross_entropy", weights=w)
    for k in oracle.TENSORS:
        for a in range(o.n_adapters):
            for l in range(o.L):
                np.testing.assert_allclose(o.G[k][a][l], o2.G[k][a][l], rtol=1e-13, atol=1e-17)


def test_dlogits_sum_to_zero():
    o, params, b = _make(7)
    h, _, _ = o.forward_hidden(b["tokens"], b["adapter_ids"])
    ell, lse = o.logprobs_from_hidden(h, b["targets"])
    g = b["dloss"].astype(np.float64)
    dz = o.dlogits(h, b["targets"].astype(np.int64), lse, g)
    assert np.max(np.abs(dz.sum(axis=1))) < 1e-13 * max(1.0, np.abs(g).max())
    # and dz at the target equals g (1 - p_target)
    p_t = np.exp(ell)
    np.testing.assert_allclose(dz[np.arange(len(g)), b["targets"]], g * (1 - p_t), rtol=1e-12, atol=1e-15)


def _grads(o):
    return [o.G[k][a][l].copy() for k in oracle.TENSORS for a in range(o.n_adapters)
            for l in range(o.L)]


def test_custom_with_minus_w_equals_cross_entropy():
    o, params, b = _make(8)
    o.forward_backward(b["tokens"], b["targets"], b["adapter_ids"], "cross_entropy", weights=b["weights"])
    o2 = oracle.Oracle(*params)
    o2.forward_backward_custom(b["tokens"], b["targets"], b["adapter_ids"], -b["weights"].astype(np.float64))
    for x, y in zip(_grads(o), _grads(o2)):
        assert np.array_equal(x, y)


def test_is_at_unit_ratio_equals_ce_and_ppo_equals_is():
    o, params, b = _make(9)
    ell = o.forward(b["tokens"], b["targets"], b["adapter_ids"])
    A = b["advantages"].astype(np.float64)
    o.forward_backward(b["tokens"], b["targets"], b["adapter_ids"], "importance_sampling",
                       advantages=A, sampler_logprobs=ell)
    o2 = oracle.Oracle(*params)
    o2.forward_backward(b["tokens"], b["targets"], b["adapter_ids"], "cross_entropy", weights=A)
    o3 = oracle.Oracle(*params)
    o3.forward_backward(b["tokens"], b["targets"], b["adapter_ids"], "ppo",
                        advantages=A, sampler_logprobs=ell, clip_eps=0.2)
    for x, y, z in zip(_grads(o), _grads(o2), _grads(o3)):
        assert np.array_equal(x, y)
        assert np.array_equal(x, z)


def test_gradients_accumulate_across_calls():
    o, params, b = _make(10)
    kw = dict(weights=b["weights"])
    o.forward_backward(b["tokens"], b["targets"], b["adapter_ids"], "cross_entropy", **kw)
    o.forward_backward(b["tokens"], b["targets"], b["adapter_ids"], "cross_entropy", **kw)
    o2 = oracle.Oracle(*params)
    o2.forward_backward(b["tokens"], b["targets"], b["adapter_ids"], "cross_entropy", **kw)
    for x, y in zip(_grads(o), _grads(o2)):
        np.testing.assert_allclose(x, 2 * y, rtol=1e-14, atol=0)


# ---------------------------------------------------------------- Adam ------

def test_adam_two_steps_exact():
    for c in golden("adam_two_steps.json")["cases"]:
        p, m, v = np.array([c["p0"]]), np.zeros(1), np.zeros(1)
        for t, (gr, st) in enumerate(zip(c["grads"], c["steps"]), start=1):
            p, m, v = oracle.adam_update(p, np.array([gr]), m, v, t, c["lr"], c["beta1"],
                                         c["beta2"], c["eps"], 0.0)
            assert abs(p[0] - st["p"]) <= 1e-15 * max(1.0, abs(st["p"]))
            assert abs(m[0] - st["m"]) <= 1e-15 * abs(st["m"]) + 1e-30
            assert abs(v[0] - st["v"]) <= 1e-14 * abs(st["v"]) + 1e-30


def test_optim_step_first_step_closed_form_and_selection():
    o, params, b = _make(11)
    ids = b["adapter_ids"].copy()
    ids[ids == 2] = 0                         # adapter 2 untouched
    o.forward_backward(b["tokens"], b["targets"], ids, "cross_entropy", weights=b["weights"])
    P0 = {k: [[x.copy() for x in row] for row in o.P[k]] for k in oracle.TENSORS}
    G0 = {k: [[x.copy() for x in row] for row in o.G[k]] for k in oracle.TENSORS}
    lr, eps = 1e-2, 1e-8
    skipped = o.optim_step(lr=lr, eps=eps)
    assert skipped == []
    assert o.step == [1, 1, 0]
    for k in oracle.TENSORS:
        for a in range(3):
            for l in range(o.L):
                if a == 2:
                    assert np.array_equal(o.P[k][a][l], P0[k][a][l])
                else:
                    G = G0[k][a][l]
                    np.testing.assert_allclose(o.P[k][a][l], P0[k][a][l] - lr * G / (np.abs(G) + eps),
                                               rtol=1e-14, atol=1e-17)
                assert not o.G[k][a][l].any()


def test_optim_step_skips_nonfinite_adapter():
    o, params, b = _make(12)
    o.forward_backward(b["tokens"], b["targets"], b["adapter_ids"], "cross_entropy", weights=b["weights"])
    o.G["B2"][1][0][0, 0] = np.nan
    P1 = [x.copy() for x in o.P["A1"][1]]
    skipped = o.optim_step()
    assert skipped == [1]
    assert o.step == [1, 0, 1]
    assert all(np.array_equal(x, y) for x, y in zip(P1, o.P["A1"][1]))
    assert not o.G["A1"][1][0].any() and not np.isnan(o.G["B2"][1][0]).any()


# ---------------------------------------------------------------- checkpoint

def test_state_file_round_trip(tmp_path):
    o, params, b = _make(13)
    o.forward_backward(b["tokens"], b["targets"], b["adapter_ids"], "cross_entropy", weights=b["weights"])
    o.optim_step(lr=1e-3)
    p = str(tmp_path / "s.bin")
    oracle.write_state_file(p, o)
    st = oracle.read_state_file(p)
    assert st["n_adapters"] == 3 and st["n_layers"] == o.L
    for a, rec in enumerate(st["adapters"]):
        assert rec["rank"] == o.ranks[a] and rec["step"] == o.step[a]
        for k in oracle.TENSORS:
            for l in range(o.L):
                np.testing.assert_array_equal(rec["P"][k][l], o.P[k][a][l].astype(np.float32))
                np.testing.assert_array_equal(rec["M"][k][l], o.M[k][a][l].astype(np.float32))
                np.testing.assert_array_equal(rec["V"][k][l], o.Vm[k][a][l].astype(np.float32))


def _ce_step(o, b, lr=1e-3):
    o.forward_backward(b["tokens"], b["targets"], b["adapter_ids"], "cross_entropy", weights=b["weights"])
    return o.optim_step(lr=lr)


def test_load_weights_only_restarts_adam(tmp_path):
    """load_state resets the history: the next step of every adapter is a
    first Adam step, whose update is the closed form -lr g / (|g| + eps)."""
    o, params, b = _make(14)
    _ce_step(o, b)
    _ce_step(o, b)
    p = str(tmp_path / "s.bin")
    oracle.write_state_file(p, o)
    q, _, _ = _make(15)                              # other base and adapters, same shapes
    q.forward_backward(b["tokens"], b["targets"], b["adapter_ids"], "cross_entropy",
                       weights=b["weights"])                    # a pending gradient ...
    oracle.load_state_file(p, q, with_optimizer=False)
    assert q.step == [0, 0, 0] and not q.touched                # ... is dropped
    assert not any(g.any() for row in q.G["B1"] for g in row)
    for a in range(3):
        np.testing.assert_array_equal(q.P["A2"][a][1], o.P["A2"][a][1].astype(np.float32))
        assert not q.M["A2"][a][1].any() and not q.Vm["B2"][a][0].any()
    P0 = {k: [[x.copy() for x in row] for row in q.P[k]] for k in oracle.TENSORS}
    q.forward_backward(b["tokens"], b["targets"], b["adapter_ids"], "cross_entropy", weights=b["weights"])
    G = {k: [[x.copy() for x in row] for row in q.G[k]] for k in oracle.TENSORS}
    q.optim_step(lr=1e-3)
    assert q.step == [1, 1, 1]
    for k in oracle.TENSORS:
        for a in range(3):
            for l in range(q.L):
                g = G[k][a][l]
                np.testing.assert_allclose(q.P[k][a][l] - P0[k][a][l], -1e-3 * g / (np.abs(g) + 1e-8),
                                           rtol=1e-9, atol=1e-15)


def test_load_with_optimizer_resumes_the_run(tmp_path):
    """load_state_with_optimizer: a run saved after two steps and resumed in a
    fresh oracle takes the same third step as the uninterrupted run (up to
    the fp32 rounding of the file), and differs from a weights-only resume."""
    o, params, b = _make(16)
    _ce_step(o, b)
    _ce_step(o, b)
    p = str(tmp_path / "s.bin")
    oracle.write_state_file(p, o)
    before = {k: [[x.copy() for x in row] for row in o.P[k]] for k in oracle.TENSORS}
    _ce_step(o, b)
    for with_opt in (True, False):
        q, _, _ = _make(16)                          # same base; adapters overwritten
        oracle.load_state_file(p, q, with_optimizer=with_opt)
        assert q.step == ([2, 2, 2] if with_opt else [0, 0, 0])
        start = {k: [[x.copy() for x in row] for row in q.P[k]] for k in oracle.TENSORS}
        _ce_step(q, b)
        worst = 0.0
        for k in oracle.TENSORS:
            for a in range(3):
                for l in range(q.L):
                    du_o = o.P[k][a][l] - before[k][a][l]
                    du_q = q.P[k][a][l] - start[k][a][l]
                    worst = max(worst, float(np.linalg.norm(du_q - du_o) / np.linalg.norm(du_o)))
        if with_opt:
            assert q.step == [3, 3, 3] and worst <= 1e-4
        else:
            assert q.step == [1, 1, 1] and worst > 1e-2


def test_load_rejects_a_mismatched_checkpoint(tmp_path):
    o, params, b = _make(18)
    p = str(tmp_path / "s.bin")
    oracle.write_state_file(p, o)
    q, _, _ = _make(18, ranks=(4, 8, 4))
    before = q.P["A1"][1][0].copy()
    with pytest.raises(ValueError):
        oracle.load_state_file(p, q, with_optimizer=True)
    np.testing.assert_array_equal(q.P["A1"][1][0], before)


def test_merged_weights_reproduce_the_adapter():
    """Export: a base whose W1, W2 are W + gamma B A of adapter a, run with
    zero adapters, gives adapter a's logprobs (and differs from the bare base)."""
    o, params, b = _make(19)
    base, ad, ranks, alphas = params
    tok, tgt = b["tokens"], b["targets"]
    for a in range(3):
        merged = {"E": base["E"], "Wout": base["Wout"],
                  "W1": [o.merged_weight(a, l, "W1") for l in range(o.L)],
                  "W2": [o.merged_weight(a, l, "W2") for l in range(o.L)]}
        zero = {k: [[np.zeros_like(x) for x in row] for row in ad[k]] for k in ad}
        q = oracle.Oracle(merged, zero, ranks, alphas)
        ids = np.full(len(tok), a)
        ref = o.forward(tok, tgt, ids)
        np.testing.assert_allclose(q.forward(tok, tgt, ids), ref, rtol=0, atol=1e-12)
        bare = oracle.Oracle(base, zero, ranks, alphas).forward(tok, tgt, ids)
        assert np.max(np.abs(bare - ref)) > 1e-3


def test_sampling_uniform_closed_form():
    """Wout = 0 makes every next-token distribution uniform: the inverse CDF
    at u is floor(u V) and its logprob -log V."""
    o, params, b = _make(20)
    o.Wout[...] = 0.0
    u = np.array([0.0, 1e-9, 0.25, 0.5 - 1e-9, 0.731, 0.999999])
    tok, ids = b["tokens"][:6], b["adapter_ids"][:6]
    nxt, lp, lo, hi = o.sample(tok, ids, u)
    assert nxt.tolist() == np.floor(u * o.V).astype(int).tolist()
    np.testing.assert_allclose(lp, -np.log(o.V), rtol=0, atol=1e-12)
    assert (lo <= u + 1e-15).all() and (u < hi).all()


def test_sampling_matches_pure_python_walk():
    """The inverse CDF equals a pure-Python walk over the softmax of the
    brute-force logits, token by token."""
    o, params, b = _make(21)
    rng = np.random.Generator(np.random.PCG64([21, 1]))
    u = rng.random(5)
    tok, ids = b["tokens"][:5], b["adapter_ids"][:5]
    nxt, lp, lo, hi = o.sample(tok, ids, u)
    base, ad, ranks, alphas = params
    for t in range(5):
        # logprobs of every target via the brute-force forward
        lps = [_brute_logprob(params, int(tok[t]), v, int(ids[t])) for v in range(o.V)]
        ps = [math.exp(x) for x in lps]
        run, pick = 0.0, o.V - 1
        for v, pv in enumerate(ps):
            run += pv
            if run > u[t]:
                pick = v
                break
        assert nxt[t] == pick
        assert abs(lp[t] - lps[pick]) < 1e-9


# ---------------------------------------------------------------- planted mistakes

def test_planted_silu_grad_error_is_caught(monkeypatch):
    monkeypatch.setattr(om, "silu_grad", lambda u: om.sigmoid(u))
    assert _fd_check("cross_entropy") > 1e-3


def test_planted_dlogits_sign_error_is_caught(monkeypatch):
    orig = om.Oracle.dlogits
    monkeypatch.setattr(om.Oracle, "dlogits", lambda self, *a: -orig(self, *a))
    assert _fd_check("custom") > 1e-3


def test_planted_adam_without_bias_correction_is_caught():
    c = golden("adam_two_steps.json")["cases"][0]

    def wrong(p, G, m, v, t, lr, b1, b2, eps, wd):
        m = b1 * m + (1 - b1) * G
        v = b2 * v + (1 - b2) * G * G
        return p - lr * m / (np.sqrt(v) + eps), m, v
    p, m, v = np.array([c["p0"]]), np.zeros(1), np.zeros(1)
    p, m, v = wrong(p, np.array([c["grads"][0]]), m, v, 1, c["lr"], 0.9, 0.999, 1e-8, 0)
    assert abs(p[0] - c["steps"][0]["p"]) > 1e-3


def test_planted_ppo_tie_rule_is_caught():
    """A PPO rule that takes the clipped branch on ties fails the golden rows."""
    g = golden("ppo_boundaries.json")

    def mutant(ell, A, s, eps):
        r = np.exp(ell - s)
        un = r * A
        cl = np.clip(r, 1.0 - eps, 1.0 + eps) * A
        return np.where(un < cl, -r * A, 0.0)
    bad = 0
    for row in g["rows"]:
        ell = np.array([math.log(row["r"])])
        r = float(np.exp(ell[0]))
        eps = {"upper": r - 1.0, "lower": 1.0 - r}.get(row.get("tie"), g["eps"])
        dl = mutant(ell, np.array([row["A"]]), np.zeros(1), eps)[0]
        if "tie" in row:
            bad += abs(dl - row["dl"]) > 1e-9
    assert bad == 4
