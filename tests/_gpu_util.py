"""GPU-test helpers: device copies of the seeded inputs and comparisons."""
import numpy as np

import oracle
import workloads as wl


def dev(x, device="cuda"):
    import torch
    x = np.ascontiguousarray(x)
    if x.dtype == np.uint16:
        return torch.from_numpy(x.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(x).to(device)


def create_handle(cfg, base, ad, max_tokens, lm_backward=None):
    """A training handle; lm_backward ("recompute" / "keep_logits") selects the
    LM-head backward mode (None keeps the library's default)."""
    import rl_step_gb300 as m
    h = m.mlora_create(cfg.vocab, cfg.d_model, cfg.d_ffn, cfg.n_layers, cfg.dtype, cfg.ranks,
                       cfg.alphas, max_tokens, dev(base["E"]), [dev(w) for w in base["W1"]],
                       [dev(w) for w in base["W2"]], dev(base["Wout"]),
                       *[[[dev(x) for x in row] for row in ad[k]]
                         for k in ("A1", "B1", "A2", "B2")])
    if lm_backward is not None:
        m.mlora_set_lm_backward(h, lm_backward)
    return h


def rel_fro(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    nr = np.linalg.norm(ref)
    return float(np.linalg.norm(x - ref) / nr) if nr > 0 else float(np.linalg.norm(x))


def loss_kwargs(kind, b, s=None):
    """Keyword arguments of both sides for one loss kind."""
    if kind == "cross_entropy":
        return {"weights": b["weights"]}
    if kind in ("importance_sampling", "ppo"):
        return {"advantages": b["advantages"], "sampler_logprobs": s, "clip_eps": b["clip_eps"]}
    return {"dloss": b["dloss"]}


def run_gpu_step(h, b, kind, s=None):
    """forward_backward (or _custom) on the GPU; returns (logprobs, loss) as numpy."""
    import rl_step_gb300 as m
    tok, tgt, ids = dev(b["tokens"]), dev(b["targets"]), dev(b["adapter_ids"])
    if kind == "custom":
        lp, loss = m.mlora_forward_backward_custom(h, tok, tgt, ids, dev(b["dloss"]))
    elif kind == "cross_entropy":
        lp, loss = m.mlora_forward_backward(h, tok, tgt, ids, kind, weights=dev(b["weights"]))
    else:
        lp, loss = m.mlora_forward_backward(h, tok, tgt, ids, kind, advantages=dev(b["advantages"]),
                                            sampler_logprobs=dev(s.astype(np.float32)),
                                            clip_eps=b["clip_eps"])
    return lp.cpu().numpy(), loss.cpu().numpy()


def run_oracle_step(o, b, kind, s=None):
    if kind == "custom":
        return o.forward_backward_custom(b["tokens"], b["targets"], b["adapter_ids"], b["dloss"])
    return o.forward_backward(b["tokens"], b["targets"], b["adapter_ids"], kind,
                              **loss_kwargs(kind, b, s))


def grad_errors(h, o, adapters, which_prefix="g"):
    """Max relative Frobenius error over the selected adapters' tensors."""
    import rl_step_gb300 as m
    worst = 0.0
    where = None
    for a in adapters:
        for l in range(o.L):
            for k in oracle.TENSORS:
                if which_prefix == "g":
                    x = m.mlora_read_adapter(h, a, l, "g" + k).cpu().numpy()
                    ref = o.G[k][a][l]
                else:
                    x = m.mlora_read_adapter(h, a, l, k).cpu().numpy()
                    ref = o.P[k][a][l]
                e = rel_fro(x, ref)
                if e > worst:
                    worst, where = e, (a, l, k)
    return worst, where
