"""CPU oracle of the multi-tenant LoRA step on a transformer block, in fp64.

TEST INFRASTRUCTURE.  Only the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this module.  The product (the CUDA
library under rl_step_gb300/) never imports, links or calls it, and this
module imports nothing from the product; the two share only the seeded input
generators in ``workloads``.

The block (tinker-ticks, "How the SGMV kernel works" and "Forward pass: what
actually happens": LoRA rides on every linear projection of a layer, the
attention projections q/k/v/o and the MLP projections gate/up/down -- seven
per layer; attention itself carries no adapter).  Written out per layer l:

    x   = rmsnorm(h) * g_attn[l]
    q   = P_q(x),  k = P_k(x),  v = P_v(x)           (grouped heads)
    q,k = rope(q, pos), rope(k, pos)
    o   = causal softmax attention of q over k, v inside each sequence
    h   = h + P_o(o)
    x   = rmsnorm(h) * g_mlp[l]
    h   = h + P_down( silu(P_gate(x)) * P_up(x) )

with P_p(x) = W_p x + gamma_a B_p,a (A_p,a x) for the token's adapter a
(Deep Dive - Tinker, "LoRA is the adaptation boundary": W' = W + gamma B A,
gamma = alpha / r), then z = Wout (rmsnorm(h) * g_final) and the target
logprob l = z[y] - logsumexp(z) (Tinker API Implementation on TPUs, section
10.3).  Losses, gradient accumulation and Adam are those of
``mlora_oracle`` (the same loss kinds, the same per-adapter optimizer).

Readings where the pages name the projections but not the block around them
(they are listed in the repository's design notes):
  * pre-norm residual block; RMSNorm y = x / sqrt(mean(x^2) + eps) * g with
    a frozen per-feature gain g, eps = 1e-6;
  * causal attention inside each sequence, heads of width hd, n_kv_heads
    key/value heads each shared by n_heads / n_kv_heads query heads (query
    head j reads key/value head j // (n_heads / n_kv_heads)); scores scaled
    by 1 / sqrt(hd);
  * rotary position embedding on q and k: for i < hd/2 the pair
    (x_i, x_{i+hd/2}) is rotated by the angle pos * theta^(-2i/hd);
  * the MLP is the gated SiLU unit silu(gate) * up;
  * no bias anywhere; the embedding and the LM head are untied and carry no
    adapter.
Sequences are given by per-token positions: a token with position 0 starts a
sequence, every other token continues the sequence of the token before it
(same adapter, position one higher).

Parity pins: tests/test_oracle_transformer_pins.py checks every function here
against finite differences, library routines (torch's scaled-dot-product
attention and rms_norm on the CPU), closed forms (single-token sequences,
position 0), invariants (causality, relative positions, B = 0, adapter
isolation, masked tokens, grouped heads versus repeated heads) and planted
mistakes.  No function is "parity unpinned".
"""
from __future__ import annotations

from typing import Iterable, List, Optional, Sequence

import numpy as np

from .mlora_oracle import _widen, adam_update, logsumexp_rows, sigmoid, silu, silu_grad, token_loss

PROJ = ("q", "k", "v", "o", "gate", "up", "down")
_TOKEN_CHUNK = 64


def proj_shapes(d: int, n_heads: int, n_kv_heads: int, head_dim: int, f: int) -> dict:
    """(out, in) of each projection's frozen weight W_p [out x in]."""
    q, kv = n_heads * head_dim, n_kv_heads * head_dim
    return {"q": (q, d), "k": (kv, d), "v": (kv, d), "o": (d, q),
            "gate": (f, d), "up": (f, d), "down": (d, f)}


# ---------------------------------------------------------------------------
# sequences, RMSNorm, rotary embedding, attention
# ---------------------------------------------------------------------------

def sequences(positions, adapter_ids) -> List[np.ndarray]:
    """Token index arrays of the batch's sequences (position 0 starts one)."""
    pos = np.asarray(positions, dtype=np.int64)
    ids = np.asarray(adapter_ids, dtype=np.int64)
    n = pos.shape[0]
    out, start = [], 0
    for t in range(n):
        if t == 0:
            if pos[0] != 0:
                raise ValueError("the first token must have position 0")
            continue
        if pos[t] == 0:
            out.append(np.arange(start, t))
            start = t
        elif pos[t] != pos[t - 1] + 1 or ids[t] != ids[t - 1]:
            raise ValueError(f"token {t} does not continue its sequence")
    if n:
        out.append(np.arange(start, n))
    return out


def rmsnorm(x, g, eps):
    """(x / sqrt(mean(x^2) + eps) * g, 1 / sqrt(mean(x^2) + eps)) per row."""
    rstd = 1.0 / np.sqrt(np.mean(x * x, axis=1) + eps)
    return x * rstd[:, None] * g[None, :], rstd


def rmsnorm_backward(x, g, rstd, dy):
    """dL/dx of y = x rstd(x) g:  rstd (g dy) - x rstd^3 mean(x g dy)."""
    gdy = dy * g[None, :]
    c = np.mean(x * gdy, axis=1)
    return rstd[:, None] * gdy - x * (rstd ** 3 * c)[:, None]


def rope_angles(positions, head_dim: int, theta: float):
    """[n x hd/2] rotation angles pos * theta^(-2i/hd)."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    inv = theta ** (-2.0 * i / head_dim)
    return np.asarray(positions, dtype=np.float64)[:, None] * inv[None, :]


def rope(x, positions, n_heads: int, head_dim: int, theta: float, inverse: bool = False):
    """Rotate every head of x [n x n_heads*hd]; inverse=True applies R^T
    (the backward of the rotation)."""
    ang = rope_angles(positions, head_dim, theta)
    c, s = np.cos(ang), np.sin(ang)
    if inverse:
        s = -s
    half = head_dim // 2
    y = np.empty_like(x)
    for hh in range(n_heads):
        a = x[:, hh * head_dim: hh * head_dim + half]
        b = x[:, hh * head_dim + half: (hh + 1) * head_dim]
        y[:, hh * head_dim: hh * head_dim + half] = a * c - b * s
        y[:, hh * head_dim + half: (hh + 1) * head_dim] = b * c + a * s
    return y


def attention(q, k, v, seqs, n_heads: int, n_kv_heads: int, head_dim: int):
    """Causal softmax attention inside each sequence; returns (o, lse) with
    lse [n x n_heads] the log-sum-exp of each row's scaled scores."""
    n = q.shape[0]
    o = np.zeros((n, n_heads * head_dim))
    lse = np.zeros((n, n_heads))
    grp = n_heads // n_kv_heads
    scale = 1.0 / np.sqrt(head_dim)
    for rows in seqs:
        T = len(rows)
        mask = np.tril(np.ones((T, T), dtype=bool))
        for hq in range(n_heads):
            hk = hq // grp
            Q = q[rows, hq * head_dim:(hq + 1) * head_dim]
            K = k[rows, hk * head_dim:(hk + 1) * head_dim]
            Vv = v[rows, hk * head_dim:(hk + 1) * head_dim]
            S = np.where(mask, (Q @ K.T) * scale, -np.inf)
            m = S.max(axis=1)
            l = m + np.log(np.exp(S - m[:, None]).sum(axis=1))
            P = np.exp(S - l[:, None])
            o[rows, hq * head_dim:(hq + 1) * head_dim] = P @ Vv
            lse[rows, hq] = l
    return o, lse


def attention_backward(q, k, v, do, seqs, n_heads: int, n_kv_heads: int, head_dim: int):
    """(dq, dk, dv) of o = softmax(q k^T / sqrt(hd), causal) v, per sequence:
    dv = P^T do, dP = do v^T, dS = P (dP - rowsum(dP P)), dq = dS k / sqrt(hd),
    dk = dS^T q / sqrt(hd); key/value heads sum over their query heads."""
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    grp = n_heads // n_kv_heads
    scale = 1.0 / np.sqrt(head_dim)
    for rows in seqs:
        T = len(rows)
        mask = np.tril(np.ones((T, T), dtype=bool))
        for hq in range(n_heads):
            hk = hq // grp
            cq = slice(hq * head_dim, (hq + 1) * head_dim)
            ck = slice(hk * head_dim, (hk + 1) * head_dim)
            Q, K, Vv, dO = q[rows, cq], k[rows, ck], v[rows, ck], do[rows, cq]
            S = np.where(mask, (Q @ K.T) * scale, -np.inf)
            P = np.exp(S - logsumexp_rows(S)[:, None])
            dv[rows, ck] += P.T @ dO
            dP = dO @ Vv.T
            dS = P * (dP - (dP * P).sum(axis=1)[:, None])
            dq[rows, cq] += dS @ K * scale
            dk[rows, ck] += dS.T @ Q * scale
    return dq, dk, dv


# ---------------------------------------------------------------------------
# the model
# ---------------------------------------------------------------------------

class TransformerOracle:
    """fp64 state of one frozen transformer base plus a pool of adapters.

    base: E [V x d], Wout [V x d], final_norm [d], attn_norm[l] [d],
          mlp_norm[l] [d], W[p][l] [out x in] for p in PROJ (bf16 bits or fp32).
    adapters: A[p][a][l] [r x in], B[p][a][l] [out x r] (fp32).
    """

    def __init__(self, base: dict, adapters: dict, ranks: Sequence[int], alphas: Sequence[float],
                 n_heads: int, n_kv_heads: int, head_dim: int, rope_theta: float = 1e6,
                 rms_eps: float = 1e-6):
        self._E = np.asarray(base["E"])
        self.V, self.d = self._E.shape
        self.Wout = _widen(base["Wout"])
        self.g_final = _widen(base["final_norm"])
        self.g_attn = [_widen(g) for g in base["attn_norm"]]
        self.g_mlp = [_widen(g) for g in base["mlp_norm"]]
        self.W = {p: [_widen(w) for w in base["W"][p]] for p in PROJ}
        self.L = len(self.g_attn)
        self.nh, self.nkv, self.hd = int(n_heads), int(n_kv_heads), int(head_dim)
        self.f = self.W["gate"][0].shape[0]
        self.theta, self.eps = float(rope_theta), float(rms_eps)
        self.n_adapters = len(ranks)
        self.ranks = [int(r) for r in ranks]
        self.alphas = [float(a) for a in alphas]
        self.gamma = [al / r for al, r in zip(self.alphas, self.ranks)]
        self.P = {}
        for p in PROJ:
            self.P["A_" + p] = [[_widen(adapters["A"][p][a][l]) for l in range(self.L)]
                                for a in range(self.n_adapters)]
            self.P["B_" + p] = [[_widen(adapters["B"][p][a][l]) for l in range(self.L)]
                                for a in range(self.n_adapters)]
        self.keys = tuple(self.P)
        zeros = lambda: {k: [[np.zeros_like(x) for x in row] for row in self.P[k]] for k in self.keys}
        self.G, self.M, self.Vm = zeros(), zeros(), zeros()
        self.step = [0] * self.n_adapters
        self.touched = set()

    # -- one adapted projection ---------------------------------------------
    def _proj(self, p, l, x, groups, save):
        y = x @ self.W[p][l].T
        vs = {}
        for a, rows in groups.items():
            vs[a] = x[rows] @ self.P["A_" + p][a][l].T                      # shrink
            y[rows] += self.gamma[a] * (vs[a] @ self.P["B_" + p][a][l].T)   # expand
        if save is not None:
            save["x_" + p] = x
            save["v_" + p] = vs
        return y

    def _proj_backward(self, p, l, dy, groups, save):
        """dL/dx of P_p; accumulates the adapter gradients of A_p and B_p."""
        dx = dy @ self.W[p][l]
        x, vs = save["x_" + p], save["v_" + p]
        for a, rows in groups.items():
            gm = self.gamma[a]
            w = gm * (dy[rows] @ self.P["B_" + p][a][l])
            dx[rows] += w @ self.P["A_" + p][a][l]
            self.G["B_" + p][a][l] += gm * (dy[rows].T @ vs[a])
            self.G["A_" + p][a][l] += w.T @ x[rows]
        return dx

    # -- forward ------------------------------------------------------------
    def forward_hidden(self, tokens, positions, adapter_ids, keep: bool = False):
        ids = np.asarray(adapter_ids, dtype=np.int64)
        pos = np.asarray(positions, dtype=np.int64)
        seqs = sequences(pos, ids)
        h = _widen(self._E[np.asarray(tokens, dtype=np.int64)])
        groups = {int(a): np.nonzero(ids == a)[0] for a in np.unique(ids)}
        saved = []
        for l in range(self.L):
            s = {} if keep else None
            h_in = h
            x1, rstd1 = rmsnorm(h_in, self.g_attn[l], self.eps)
            q = rope(self._proj("q", l, x1, groups, s), pos, self.nh, self.hd, self.theta)
            k = rope(self._proj("k", l, x1, groups, s), pos, self.nkv, self.hd, self.theta)
            v = self._proj("v", l, x1, groups, s)
            o, _ = attention(q, k, v, seqs, self.nh, self.nkv, self.hd)
            h_mid = h_in + self._proj("o", l, o, groups, s)
            x2, rstd2 = rmsnorm(h_mid, self.g_mlp[l], self.eps)
            gate = self._proj("gate", l, x2, groups, s)
            up = self._proj("up", l, x2, groups, s)
            act = silu(gate) * up
            h = h_mid + self._proj("down", l, act, groups, s)
            if keep:
                s.update({"h_in": h_in, "rstd1": rstd1, "q": q, "k": k, "v": v,
                          "h_mid": h_mid, "rstd2": rstd2, "gate": gate, "up": up})
                saved.append(s)
        xf, rstdf = rmsnorm(h, self.g_final, self.eps)
        return xf, {"h": h, "rstd": rstdf, "layers": saved, "seqs": seqs, "pos": pos}, groups

    def logprobs_from_hidden(self, xf, targets):
        y = np.asarray(targets, dtype=np.int64)
        n = xf.shape[0]
        ell, lse = np.empty(n), np.empty(n)
        for c0 in range(0, n, _TOKEN_CHUNK):
            c1 = min(n, c0 + _TOKEN_CHUNK)
            z = xf[c0:c1] @ self.Wout.T
            lse[c0:c1] = logsumexp_rows(z)
            ell[c0:c1] = z[np.arange(c1 - c0), y[c0:c1]] - lse[c0:c1]
        return ell, lse

    def forward(self, tokens, targets, positions, adapter_ids) -> np.ndarray:
        """Target-token logprobs; no state change."""
        xf, _, _ = self.forward_hidden(tokens, positions, adapter_ids)
        return self.logprobs_from_hidden(xf, targets)[0]

    # -- backward -----------------------------------------------------------
    def forward_backward(self, tokens, targets, positions, adapter_ids, kind: str, *,
                         weights=None, advantages=None, sampler_logprobs=None,
                         clip_eps: float = 0.2, dloss=None) -> dict:
        """Forward, loss, adapter-only backward; gradients accumulate."""
        y = np.asarray(targets, dtype=np.int64)
        xf, st, groups = self.forward_hidden(tokens, positions, adapter_ids, keep=True)
        ell, lse = self.logprobs_from_hidden(xf, y)
        val, g = token_loss(kind, ell, weights=weights, advantages=advantages,
                            sampler_logprobs=sampler_logprobs, clip_eps=clip_eps, dloss=dloss)
        loss = np.zeros(self.n_adapters)
        for a, rows in groups.items():
            loss[a] = val[rows].sum()

        n = xf.shape[0]
        dxf = np.empty_like(xf)
        for c0 in range(0, n, _TOKEN_CHUNK):
            c1 = min(n, c0 + _TOKEN_CHUNK)
            z = xf[c0:c1] @ self.Wout.T
            dz = -g[c0:c1, None] * np.exp(z - lse[c0:c1, None])
            dz[np.arange(c1 - c0), y[c0:c1]] += g[c0:c1]
            dxf[c0:c1] = dz @ self.Wout
        dh = rmsnorm_backward(st["h"], self.g_final, st["rstd"], dxf)
        pos, seqs = st["pos"], st["seqs"]
        for l in reversed(range(self.L)):
            s = st["layers"][l]
            # h = h_mid + P_down(silu(gate) * up)
            dact = self._proj_backward("down", l, dh, groups, s)
            dgate = dact * s["up"] * silu_grad(s["gate"])
            dup = dact * silu(s["gate"])
            dx2 = self._proj_backward("gate", l, dgate, groups, s)
            dx2 += self._proj_backward("up", l, dup, groups, s)
            dh = dh + rmsnorm_backward(s["h_mid"], self.g_mlp[l], s["rstd2"], dx2)
            # h_mid = h_in + P_o(attention(rope(P_q x), rope(P_k x), P_v x))
            do = self._proj_backward("o", l, dh, groups, s)
            dq, dk, dv = attention_backward(s["q"], s["k"], s["v"], do, seqs,
                                            self.nh, self.nkv, self.hd)
            dq = rope(dq, pos, self.nh, self.hd, self.theta, inverse=True)
            dk = rope(dk, pos, self.nkv, self.hd, self.theta, inverse=True)
            dx1 = self._proj_backward("q", l, dq, groups, s)
            dx1 += self._proj_backward("k", l, dk, groups, s)
            dx1 += self._proj_backward("v", l, dv, groups, s)
            dh = dh + rmsnorm_backward(s["h_in"], self.g_attn[l], s["rstd1"], dx1)
        self.touched.update(groups.keys())
        return {"logprobs": ell, "loss_per_adapter": loss, "g": g}

    def forward_backward_custom(self, tokens, targets, positions, adapter_ids, dloss) -> dict:
        """Backpropagate sum_t g_t l_t with the caller's g = dC/dl."""
        return self.forward_backward(tokens, targets, positions, adapter_ids, "custom", dloss=dloss)

    # -- optimizer ----------------------------------------------------------
    def optim_step(self, lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0,
                   adapters: Optional[Iterable[int]] = None) -> List[int]:
        """Adam on the selected adapters (default: those touched); returns skipped ids."""
        sel = sorted(self.touched) if adapters is None else sorted(set(int(a) for a in adapters))
        skipped = []
        for a in sel:
            finite = all(np.isfinite(self.G[k][a][l]).all() for k in self.keys for l in range(self.L))
            if finite:
                t = self.step[a] + 1
                for k in self.keys:
                    for l in range(self.L):
                        p, m, v = adam_update(self.P[k][a][l], self.G[k][a][l], self.M[k][a][l],
                                              self.Vm[k][a][l], t, lr, beta1, beta2, eps, weight_decay)
                        self.P[k][a][l], self.M[k][a][l], self.Vm[k][a][l] = p, m, v
                self.step[a] = t
            else:
                skipped.append(a)
            for k in self.keys:
                for l in range(self.L):
                    self.G[k][a][l][...] = 0.0
            self.touched.discard(a)
        return skipped
