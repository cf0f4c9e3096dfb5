"""The transformer-block definition evaluated in fp64 with only the values the
CUDA path stores between kernels rounded to bf16 (test infrastructure).

It derives the tolerances of the transformer-block parity tests: how far from
the exact fp64 result any implementation that stores these activations in
bf16 (and computes everything else exactly) must land.  It is the oracle's
arithmetic (oracle/transformer_oracle.py) with a rounding inserted at each
storage point; it imports nothing from the CUDA path.

Rounded to bf16 (round to nearest even): the normalised inputs of the
projections, q / k / v before and after the rotary embedding, the attention
output, the kept gate / up values and silu(gate) * up, the final normalised
hidden state, every LoRA shrink output gamma A x and backward shrink
gamma B^T dy, the LM head's dL/dz, the residual gradient as a GEMM input, the
gated-MLP input gradients, dL/dO and dL/d(q, k, v) before and after the
inverse rotation.  Everything else (residual stream, norms, softmax,
accumulations) stays fp64.
"""
import numpy as np

import oracle.transformer_oracle as to
from oracle.mlora_oracle import silu, silu_grad, token_loss
from workloads import bf16_bits_to_f32, f32_to_bf16_bits


def bf(x):
    """Round to bf16 and widen back (exact widening)."""
    return bf16_bits_to_f32(f32_to_bf16_bits(np.asarray(x, np.float32))).astype(np.float64)


class BF16StorageModel(to.TransformerOracle):
    """TransformerOracle with bf16 rounding at the CUDA path's storage points.

    round_lm_input = False leaves the final normalised hidden state (the LM
    head's input) exact, to separate its share of the logprob error from the
    layers' (at the 8B widths, four layers, three 48-token prefixes: 0.057 max
    logprob error with it rounded, 0.059 without -- the layers dominate)."""

    round_lm_input = True

    def _proj(self, p, l, x, groups, save):
        y = x @ self.W[p][l].T
        vs = {}
        for a, rows in groups.items():
            vs[a] = bf(self.gamma[a] * (x[rows] @ self.P["A_" + p][a][l].T))
            y[rows] += vs[a] @ self.P["B_" + p][a][l].T
        if save is not None:
            save["x_" + p] = x
            save["v_" + p] = vs
        return y

    def _proj_backward(self, p, l, dy, groups, save):
        dx = dy @ self.W[p][l]
        x, vs = save["x_" + p], save["v_" + p]
        for a, rows in groups.items():
            w = bf(self.gamma[a] * (dy[rows] @ self.P["B_" + p][a][l]))
            dx[rows] += w @ self.P["A_" + p][a][l]
            self.G["B_" + p][a][l] += dy[rows].T @ vs[a]
            self.G["A_" + p][a][l] += w.T @ x[rows]
        return dx

    def forward_hidden(self, tokens, positions, adapter_ids, keep=False):
        ids = np.asarray(adapter_ids, np.int64)
        pos = np.asarray(positions, np.int64)
        seqs = to.sequences(pos, ids)
        h = to._widen(self._E[np.asarray(tokens, np.int64)])
        groups = {int(a): np.nonzero(ids == a)[0] for a in np.unique(ids)}
        saved = []
        for l in range(self.L):
            s = {} if keep else None
            h_in = h
            x1, rstd1 = to.rmsnorm(h_in, self.g_attn[l], self.eps)
            x1 = bf(x1)
            q = bf(to.rope(bf(self._proj("q", l, x1, groups, s)), pos, self.nh, self.hd, self.theta))
            k = bf(to.rope(bf(self._proj("k", l, x1, groups, s)), pos, self.nkv, self.hd, self.theta))
            v = bf(self._proj("v", l, x1, groups, s))
            o, _ = to.attention(q, k, v, seqs, self.nh, self.nkv, self.hd)
            o = bf(o)
            h_mid = h_in + self._proj("o", l, o, groups, s)
            x2, rstd2 = to.rmsnorm(h_mid, self.g_mlp[l], self.eps)
            x2 = bf(x2)
            gate = self._proj("gate", l, x2, groups, s)
            up = self._proj("up", l, x2, groups, s)
            act = bf(silu(gate) * up)
            h = h_mid + self._proj("down", l, act, groups, s)
            if keep:
                s.update({"h_in": h_in, "rstd1": rstd1, "q": q, "k": k, "v": v, "h_mid": h_mid,
                          "rstd2": rstd2, "gate": bf(gate), "up": bf(up)})
                saved.append(s)
        xf, rstdf = to.rmsnorm(h, self.g_final, self.eps)
        if self.round_lm_input:
            xf = bf(xf)
        return xf, {"h": h, "rstd": rstdf, "layers": saved, "seqs": seqs, "pos": pos}, groups

    def forward_backward(self, tokens, targets, positions, adapter_ids, kind, **kw):
        y = np.asarray(targets, np.int64)
        xf, st, groups = self.forward_hidden(tokens, positions, adapter_ids, keep=True)
        ell, lse = self.logprobs_from_hidden(xf, y)
        val, g = token_loss(kind, ell, **kw)
        z = xf @ self.Wout.T
        dz = -g[:, None] * np.exp(z - lse[:, None])
        dz[np.arange(len(y)), y] += g
        dh = to.rmsnorm_backward(st["h"], self.g_final, st["rstd"], bf(dz) @ self.Wout)
        pos, seqs = st["pos"], st["seqs"]
        for l in reversed(range(self.L)):
            s = st["layers"][l]
            dact = self._proj_backward("down", l, bf(dh), groups, s)
            dgate = bf(dact * s["up"] * silu_grad(s["gate"]))
            dup = bf(dact * silu(s["gate"]))
            dx2 = self._proj_backward("gate", l, dgate, groups, s) + self._proj_backward("up", l, dup, groups, s)
            dh = dh + to.rmsnorm_backward(s["h_mid"], self.g_mlp[l], s["rstd2"], dx2)
            do = bf(self._proj_backward("o", l, bf(dh), groups, s))
            dq, dk, dv = to.attention_backward(s["q"], s["k"], s["v"], do, seqs, self.nh, self.nkv, self.hd)
            dq = bf(to.rope(bf(dq), pos, self.nh, self.hd, self.theta, inverse=True))
            dk = bf(to.rope(bf(dk), pos, self.nkv, self.hd, self.theta, inverse=True))
            dx1 = (self._proj_backward("q", l, dq, groups, s) + self._proj_backward("k", l, dk, groups, s)
                   + self._proj_backward("v", l, bf(dv), groups, s))
            dh = dh + to.rmsnorm_backward(s["h_in"], self.g_attn[l], s["rstd1"], dx1)
        self.touched.update(groups.keys())
        return {"logprobs": ell}
