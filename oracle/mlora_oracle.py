"""CPU oracle for one multi-tenant LoRA training step, in fp64.

TEST INFRASTRUCTURE.  Only the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this module.  The product (the CUDA
library under rl_step_gb300/) never imports, links or calls it, and this
module imports nothing from the product; the two share only the seeded input
generators in ``workloads``.

What it computes -- the plain definitions, written out:

* Routing (tinker-ticks, "How the SGMV kernel works"): all tenants' tokens
  are flattened into one matrix and a segment index records which adapter
  owns each row.  Here: a stable sort of token positions by adapter id, the
  exclusive prefix of per-adapter counts, and the same prefix after every
  segment is padded up to a multiple of the routing tile height TILE_M.
* Model (the workload definition: token embedding, L residual SiLU-MLP
  blocks h += W2 silu(W1 h), untied LM head).  Every W1 and W2 carries a LoRA
  update W' = W + gamma B A with gamma = alpha / r (Deep Dive - Tinker, "LoRA
  is the adaptation boundary" and "Checkpoints and export paths"), applied
  per token with the token's own adapter as the shrink/expand pair
  x -> A x -> gamma B (A x) (tinker-ticks, "Forward pass: what actually
  happens").
* Target logprob (Tinker API Implementation on TPUs, section 10, "3 - Never
  materialize a log-softmax"): l = z[y] - logsumexp(z), with the stable
  logsumexp m + log sum exp(z - m), m = max z.
* Losses, summed over tokens with no normalisation (Deep Dive - Tinker,
  "The RL datum shape"):
    cross_entropy        L = -sum w_t l_t
    importance_sampling  L = -sum r_t A_t,  r_t = exp(l_t - s_t)
    ppo                  L = -sum min(r_t A_t, clip(r_t, 1-eps, 1+eps) A_t)
    custom               surrogate sum g_t l_t with the caller's g_t = dC/dl_t
                         (Deep Dive - Tinker, same section; Telegram note on
                         forward_backward_custom)
  A token whose loss inputs, logprob or ratio are not finite contributes
  neither value nor gradient (Tinker API Implementation on TPUs, section 12,
  "The instability I have not solved").
* Gradients: adapter factors only; the base stays frozen (Tinker API
  Implementation on TPUs, section 4: only adapter gradients exist).  They
  accumulate across forward_backward calls until optim_step consumes them
  (Deep Dive - Tinker, "optim_step advances adapter state").
* optim_step: per-adapter Adam with bias correction and decoupled weight
  decay (default 0), one step counter per adapter, applied to adapters that
  received tokens since the previous step; an adapter whose accumulated
  gradient is not finite is skipped and reported (same two sources).

Readings where the pages are silent are listed in the repository's design
notes; the ones that shape arithmetic here: the PPO minimum picks the
unclipped branch on ties, so its gradient is -r A whenever r A <= clip(r) A
and 0 otherwise; Adam uses beta1=0.9, beta2=0.999, eps=1e-8 outside the
square root; a skipped adapter keeps p, m, v and its step count and its
gradient is consumed.

Parity pins: every function here is checked against closed forms,
invariants, library routines, brute force or the pages' worked examples by
tests/test_oracle_*.py.  No function is "parity unpinned".
"""
from __future__ import annotations

import struct
from typing import Dict, Iterable, List, Optional, Sequence

import numpy as np

TILE_M = 128          # routing tile height; equals the library's MLORA_TILE_M
LOSS_KINDS = ("cross_entropy", "importance_sampling", "ppo", "custom")
_TOKEN_CHUNK = 64     # tokens per logits block (memory bound only)


# ---------------------------------------------------------------------------
# routing
# ---------------------------------------------------------------------------

def routing(adapter_ids, n_adapters: int, tile_m: int = TILE_M) -> dict:
    """Stable grouping of token positions by adapter.

    perm[i]     position (in the batch) of the i-th token in adapter order;
                tokens of one adapter keep their batch order.
    seg_off[a]  first index in perm of adapter a; seg_off[n_adapters] = N.
    pad_off[a]  the same offset once each adapter's segment is padded to a
                multiple of tile_m rows.
    tile_ad[j]  adapter owning padded row tile j (tile_m rows each).
    """
    a = np.asarray(adapter_ids, dtype=np.int64)
    if a.size and (a.min() < 0 or a.max() >= n_adapters):
        raise ValueError("adapter id out of range")
    perm = np.argsort(a, kind="stable").astype(np.int64)
    counts = np.bincount(a, minlength=n_adapters).astype(np.int64)
    seg_off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    tiles = (counts + tile_m - 1) // tile_m
    pad_off = np.concatenate([[0], np.cumsum(tiles * tile_m)]).astype(np.int64)
    tile_ad = np.repeat(np.arange(n_adapters, dtype=np.int64), tiles)
    return {"perm": perm, "seg_off": seg_off, "pad_off": pad_off,
            "tile_ad": tile_ad, "counts": counts}


# ---------------------------------------------------------------------------
# elementwise pieces
# ---------------------------------------------------------------------------

def sigmoid(u):
    return 1.0 / (1.0 + np.exp(-u))


def silu(u):
    return u * sigmoid(u)


def silu_grad(u):
    """d/du [u sigmoid(u)] = sigmoid(u) (1 + u (1 - sigmoid(u)))."""
    s = sigmoid(u)
    return s * (1.0 + u * (1.0 - s))


def logsumexp_rows(z):
    """Stable row-wise logsumexp: m + log sum exp(z - m), m = row max."""
    m = z.max(axis=1)
    return m + np.log(np.exp(z - m[:, None]).sum(axis=1))


def token_loss(kind: str, ell, *, weights=None, advantages=None,
               sampler_logprobs=None, clip_eps: float = 0.2, dloss=None):
    """Per-token loss value and dL/dl for one of the four loss kinds.

    Returns (value_t, g_t) as fp64 arrays; tokens with non-finite inputs get
    value 0 and g 0.
    """
    ell = np.asarray(ell, dtype=np.float64)
    n = ell.shape[0]
    with np.errstate(over="ignore", invalid="ignore"):
        if kind == "cross_entropy":
            w = np.asarray(weights, dtype=np.float64)
            val = -w * ell
            g = -w
            ok = np.isfinite(w) & np.isfinite(ell)
        elif kind in ("importance_sampling", "ppo"):
            A = np.asarray(advantages, dtype=np.float64)
            s = np.asarray(sampler_logprobs, dtype=np.float64)
            r = np.exp(ell - s)
            unclipped = r * A
            if kind == "importance_sampling":
                val = -unclipped
                g = -r * A
            else:
                clipped = np.clip(r, 1.0 - clip_eps, 1.0 + clip_eps) * A
                val = -np.minimum(unclipped, clipped)
                g = np.where(unclipped <= clipped, -r * A, 0.0)
            ok = np.isfinite(A) & np.isfinite(s) & np.isfinite(ell) & np.isfinite(r)
        elif kind == "custom":
            c = np.asarray(dloss, dtype=np.float64)
            val = c * ell
            g = c.copy()
            ok = np.isfinite(c) & np.isfinite(ell)
        else:
            raise ValueError(f"unknown loss kind {kind!r}")
        ok &= np.isfinite(val) & np.isfinite(g)
    val = np.where(ok, val, 0.0)
    g = np.where(ok, g, 0.0)
    assert val.shape == (n,) and g.shape == (n,)
    return val, g


def adam_update(p, G, m, v, t: int, lr, beta1, beta2, eps, weight_decay):
    """One Adam step at step count t (t >= 1) on fp64 arrays; returns p, m, v."""
    m = beta1 * m + (1.0 - beta1) * G
    v = beta2 * v + (1.0 - beta2) * G * G
    m_hat = m / (1.0 - beta1 ** t)
    v_hat = v / (1.0 - beta2 ** t)
    p = p - lr * (m_hat / (np.sqrt(v_hat) + eps) + weight_decay * p)
    return p, m, v


# ---------------------------------------------------------------------------
# the model
# ---------------------------------------------------------------------------

def _widen(x) -> np.ndarray:
    """bf16 bit patterns (uint16) or fp32 values -> fp64 values (exact)."""
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


TENSORS = ("A1", "B1", "A2", "B2")


class Oracle:
    """fp64 state of one frozen base plus a pool of LoRA adapters."""

    def __init__(self, base: dict, adapters: dict, ranks: Sequence[int],
                 alphas: Sequence[float]):
        self._E = np.asarray(base["E"])            # widened per gathered row
        self.V, self.d = self._E.shape
        self.Wout = _widen(base["Wout"])
        self.W1 = [_widen(w) for w in base["W1"]]
        self.W2 = [_widen(w) for w in base["W2"]]
        self.L = len(self.W1)
        self.f = self.W1[0].shape[0]
        self.n_adapters = len(ranks)
        self.ranks = [int(r) for r in ranks]
        self.alphas = [float(a) for a in alphas]
        self.gamma = [al / r for al, r in zip(self.alphas, self.ranks)]
        self.P = {k: [[_widen(adapters[k][a][l]) for l in range(self.L)]
                      for a in range(self.n_adapters)] for k in TENSORS}
        self.G = {k: [[np.zeros_like(x) for x in row] for row in self.P[k]] for k in TENSORS}
        self.M = {k: [[np.zeros_like(x) for x in row] for row in self.P[k]] for k in TENSORS}
        self.Vm = {k: [[np.zeros_like(x) for x in row] for row in self.P[k]] for k in TENSORS}
        self.step = [0] * self.n_adapters
        self.touched = set()

    # -- forward ------------------------------------------------------------
    def embed(self, tokens) -> np.ndarray:
        return _widen(self._E[np.asarray(tokens, dtype=np.int64)])

    def forward_hidden(self, tokens, adapter_ids, keep: bool = False):
        """Final hidden states; with keep=True also every layer's saved values."""
        ids = np.asarray(adapter_ids, dtype=np.int64)
        h = self.embed(tokens)
        groups = {int(a): np.nonzero(ids == a)[0] for a in np.unique(ids)}
        saved = []
        for l in range(self.L):
            h_in = h
            u = h_in @ self.W1[l].T
            v1 = {}
            for a, rows in groups.items():
                v1[a] = h_in[rows] @ self.P["A1"][a][l].T                  # shrink
                u[rows] += self.gamma[a] * (v1[a] @ self.P["B1"][a][l].T)  # expand
            act = silu(u)
            y = act @ self.W2[l].T
            v2 = {}
            for a, rows in groups.items():
                v2[a] = act[rows] @ self.P["A2"][a][l].T
                y[rows] += self.gamma[a] * (v2[a] @ self.P["B2"][a][l].T)
            h = h_in + y
            if keep:
                saved.append({"h_in": h_in, "u": u, "act": act, "v1": v1, "v2": v2})
        return h, saved, groups

    def logits(self, h) -> np.ndarray:
        return h @ self.Wout.T

    def logprobs_from_hidden(self, h, targets):
        """(l, lse) per token, blockwise over tokens only."""
        y = np.asarray(targets, dtype=np.int64)
        n = h.shape[0]
        ell = np.empty(n)
        lse = np.empty(n)
        for c0 in range(0, n, _TOKEN_CHUNK):
            c1 = min(n, c0 + _TOKEN_CHUNK)
            z = self.logits(h[c0:c1])
            lse[c0:c1] = logsumexp_rows(z)
            ell[c0:c1] = z[np.arange(c1 - c0), y[c0:c1]] - lse[c0:c1]
        return ell, lse

    def forward(self, tokens, targets, adapter_ids) -> np.ndarray:
        """Target-token logprobs; no state change."""
        h, _, _ = self.forward_hidden(tokens, adapter_ids)
        return self.logprobs_from_hidden(h, targets)[0]

    def next_token_cdf(self, tokens, adapter_ids) -> np.ndarray:
        """Cumulative next-token distribution per row, [n x V] fp64: the
        running sum of softmax(z) in vocabulary order (Deep Dive - Tinker,
        "sample returns evidence for learning": the sampler returns generated
        token ids and one logprob per generated token)."""
        h, _, _ = self.forward_hidden(tokens, adapter_ids)
        z = self.logits(h)
        p = np.exp(z - logsumexp_rows(z)[:, None])
        return np.cumsum(p, axis=1)

    def sample(self, tokens, adapter_ids, uniforms):
        """Inverse-CDF sampling at temperature 1: for row t the smallest id v
        with CDF(v) > u_t (the last id when rounding leaves CDF(V-1) <= u_t).
        Returns (next ids, their logprobs, CDF(v-1), CDF(v))."""
        cdf = self.next_token_cdf(tokens, adapter_ids)
        u = np.asarray(uniforms, dtype=np.float64)
        n, V = cdf.shape
        nxt = np.empty(n, dtype=np.int64)
        lo = np.empty(n)
        hi = np.empty(n)
        for t in range(n):
            v = int(np.searchsorted(cdf[t], u[t], side="right"))
            v = min(v, V - 1)
            nxt[t] = v
            lo[t] = cdf[t, v - 1] if v > 0 else 0.0
            hi[t] = cdf[t, v]
        lp = np.log(hi - lo)
        return nxt, lp, lo, hi

    def merged_weight(self, a: int, l: int, which: str) -> np.ndarray:
        """W' = W + gamma B A for W1 or W2 of layer l with adapter a's factors
        (Deep Dive - Tinker, "Checkpoints and export paths"), in fp64."""
        if which == "W1":
            return self.W1[l] + self.gamma[a] * (self.P["B1"][a][l] @ self.P["A1"][a][l])
        return self.W2[l] + self.gamma[a] * (self.P["B2"][a][l] @ self.P["A2"][a][l])

    # -- backward -----------------------------------------------------------
    def dlogits(self, h_block, y_block, lse_block, g_block) -> np.ndarray:
        """dL/dz = g (onehot(y) - softmax(z)) for a block of tokens."""
        z = self.logits(h_block)
        p = np.exp(z - lse_block[:, None])
        dz = -g_block[:, None] * p
        dz[np.arange(len(y_block)), y_block] += g_block
        return dz

    def forward_backward(self, tokens, targets, adapter_ids, kind: str, *,
                         weights=None, advantages=None, sampler_logprobs=None,
                         clip_eps: float = 0.2, dloss=None) -> dict:
        """Forward, loss, adapter-only backward; gradients accumulate.

        Returns dict(logprobs, loss_per_adapter, g).
        """
        y = np.asarray(targets, dtype=np.int64)
        ids = np.asarray(adapter_ids, dtype=np.int64)
        h, saved, groups = self.forward_hidden(tokens, ids, keep=True)
        ell, lse = self.logprobs_from_hidden(h, y)
        val, g = token_loss(kind, ell, weights=weights, advantages=advantages,
                            sampler_logprobs=sampler_logprobs, clip_eps=clip_eps,
                            dloss=dloss)
        loss = np.zeros(self.n_adapters)
        for a, rows in groups.items():
            loss[a] = val[rows].sum()

        n = h.shape[0]
        dh = np.empty_like(h)
        for c0 in range(0, n, _TOKEN_CHUNK):
            c1 = min(n, c0 + _TOKEN_CHUNK)
            dz = self.dlogits(h[c0:c1], y[c0:c1], lse[c0:c1], g[c0:c1])
            dh[c0:c1] = dz @ self.Wout

        for l in reversed(range(self.L)):
            s = saved[l]
            # h_out = h_in + W2 act + gamma B2 (A2 act)
            dact = dh @ self.W2[l]
            for a, rows in groups.items():
                gm = self.gamma[a]
                w2 = gm * (dh[rows] @ self.P["B2"][a][l])           # [n, r]
                dact[rows] += w2 @ self.P["A2"][a][l]
                self.G["B2"][a][l] += gm * (dh[rows].T @ s["v2"][a])
                self.G["A2"][a][l] += w2.T @ s["act"][rows]
            du = dact * silu_grad(s["u"])
            # u = W1 h_in + gamma B1 (A1 h_in)
            dh_in = dh + du @ self.W1[l]
            for a, rows in groups.items():
                gm = self.gamma[a]
                w1 = gm * (du[rows] @ self.P["B1"][a][l])
                dh_in[rows] += w1 @ self.P["A1"][a][l]
                self.G["B1"][a][l] += gm * (du[rows].T @ s["v1"][a])
                self.G["A1"][a][l] += w1.T @ s["h_in"][rows]
            dh = dh_in
        self.touched.update(groups.keys())
        return {"logprobs": ell, "loss_per_adapter": loss, "g": g}

    def forward_backward_custom(self, tokens, targets, adapter_ids, dloss) -> dict:
        """Backpropagate sum_t g_t l_t with the caller's g = dC/dl."""
        return self.forward_backward(tokens, targets, adapter_ids, "custom", dloss=dloss)

    # -- optimizer ----------------------------------------------------------
    def optim_step(self, lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8,
                   weight_decay=0.0, adapters: Optional[Iterable[int]] = None) -> List[int]:
        """Adam on the selected adapters (default: those touched); returns skipped ids."""
        sel = sorted(self.touched) if adapters is None else sorted(set(int(a) for a in adapters))
        skipped = []
        for a in sel:
            finite = all(np.isfinite(self.G[k][a][l]).all()
                         for k in TENSORS for l in range(self.L))
            if finite:
                t = self.step[a] + 1
                for k in TENSORS:
                    for l in range(self.L):
                        p, m, v = adam_update(self.P[k][a][l], self.G[k][a][l],
                                              self.M[k][a][l], self.Vm[k][a][l], t,
                                              lr, beta1, beta2, eps, weight_decay)
                        self.P[k][a][l], self.M[k][a][l], self.Vm[k][a][l] = p, m, v
                self.step[a] = t
            else:
                skipped.append(a)
            for k in TENSORS:
                for l in range(self.L):
                    self.G[k][a][l][...] = 0.0
            self.touched.discard(a)
        return skipped


# ---------------------------------------------------------------------------
# checkpoint file format (save_state)
# ---------------------------------------------------------------------------
#
# Little-endian.  Header: 8-byte magic b"MLORASTA", then u32 version (1),
# u32 n_adapters, u32 n_layers, u32 d_model, u32 d_ffn, u32 0 (reserved).
# Then for each adapter a: u32 rank, f32 alpha, u64 step count, followed by
# three groups -- weights, first moments, second moments -- each holding, for
# every layer l, A1 [r x d], B1 [f x r], A2 [r x f], B2 [d x r] as fp32
# row-major arrays.

MAGIC = b"MLORASTA"


def write_state_file(path: str, o: "Oracle") -> None:
    """Write the oracle's adapter state in the checkpoint format above."""
    with open(path, "wb") as fh:
        fh.write(MAGIC)
        fh.write(struct.pack("<6I", 1, o.n_adapters, o.L, o.d, o.f, 0))
        for a in range(o.n_adapters):
            fh.write(struct.pack("<IfQ", o.ranks[a], o.alphas[a], o.step[a]))
            for group in (o.P, o.M, o.Vm):
                for l in range(o.L):
                    for k in TENSORS:
                        fh.write(np.ascontiguousarray(group[k][a][l], dtype="<f4").tobytes())


def read_state_file(path: str) -> dict:
    """Parse a checkpoint file into nested dicts of fp32 arrays."""
    with open(path, "rb") as fh:
        buf = fh.read()
    if buf[:8] != MAGIC:
        raise ValueError("not an adapter checkpoint")
    version, n_ad, L, d, f, _ = struct.unpack_from("<6I", buf, 8)
    if version != 1:
        raise ValueError(f"unsupported checkpoint version {version}")
    off = 8 + 24
    out = {"n_adapters": n_ad, "n_layers": L, "d_model": d, "d_ffn": f, "adapters": []}
    for a in range(n_ad):
        r, alpha, step = struct.unpack_from("<IfQ", buf, off)
        off += 16
        shapes = {"A1": (r, d), "B1": (f, r), "A2": (r, f), "B2": (d, r)}
        rec = {"rank": r, "alpha": alpha, "step": step}
        for gname in ("P", "M", "V"):
            grp = {k: [] for k in TENSORS}
            for l in range(L):
                for k in TENSORS:
                    cnt = shapes[k][0] * shapes[k][1]
                    arr = np.frombuffer(buf, dtype="<f4", count=cnt, offset=off).reshape(shapes[k])
                    off += 4 * cnt
                    grp[k].append(arr.astype(np.float32))
            rec[gname] = grp
        out["adapters"].append(rec)
    if off != len(buf):
        raise ValueError("trailing bytes in checkpoint")
    return out


def load_state_file(path: str, o: "Oracle", with_optimizer: bool) -> None:
    """Restore the oracle's adapters from a checkpoint file.

    Deep Dive - Tinker, "optim_step advances adapter state": loading the
    weights alone resets the optimizer history, loading with the optimizer
    restores the saved moments; "save_state creates a recovery point" names
    the two calls load_state and load_state_with_optimizer.  Reading taken
    where the page is silent: a reset history means zero moments and a step
    count of zero (the next Adam step is the first, with its bias
    correction), and any gradient accumulated before the load is dropped.
    The file must describe the same adapters (count, layers, widths, ranks,
    alphas); otherwise ValueError and the oracle is unchanged.
    """
    st = read_state_file(path)
    if (st["n_adapters"], st["n_layers"], st["d_model"], st["d_ffn"]) != (o.n_adapters, o.L, o.d, o.f):
        raise ValueError("checkpoint shape does not match")
    for a, rec in enumerate(st["adapters"]):
        if rec["rank"] != o.ranks[a] or np.float32(rec["alpha"]) != np.float32(o.alphas[a]):
            raise ValueError(f"adapter {a}: rank or alpha does not match")
    for a, rec in enumerate(st["adapters"]):
        for k in TENSORS:
            for l in range(o.L):
                o.P[k][a][l] = rec["P"][k][l].astype(np.float64)
                if with_optimizer:
                    o.M[k][a][l] = rec["M"][k][l].astype(np.float64)
                    o.Vm[k][a][l] = rec["V"][k][l].astype(np.float64)
                else:
                    o.M[k][a][l] = np.zeros_like(o.P[k][a][l])
                    o.Vm[k][a][l] = np.zeros_like(o.P[k][a][l])
                o.G[k][a][l] = np.zeros_like(o.P[k][a][l])
        o.step[a] = int(rec["step"]) if with_optimizer else 0
    o.touched = set()
