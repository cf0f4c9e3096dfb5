"""Python binding of the transformer-block entry points of libmlora.so
(include/mlora_tf.h).  Argument marshalling only: every step runs in the
library's CUDA kernels; PyTorch provides device memory and streams.

    h = tf_create(cfg fields, base, adapters, max_tokens)
    tf_forward(h, tokens, targets, positions, adapter_ids)                -> logprobs
    tf_forward_backward(h, tokens, targets, positions, adapter_ids, kind, ...)
    tf_forward_backward_custom(h, tokens, targets, positions, adapter_ids, dloss)
    tf_optim_step(h, lr=..., ...)                                         -> skipped
"""
from __future__ import annotations

import ctypes
from ctypes import POINTER, c_double, c_float, c_int32, c_int64, c_void_p
from typing import Optional, Sequence

from . import LOSS_KINDS, _Adam, _check, _LossInputs, _ptr, _stream, load_library

__all__ = ["PROJ", "TF_PROF_CLASSES", "TfHandle", "tf_create", "tf_destroy", "tf_forward",
           "tf_forward_backward", "tf_forward_backward_custom", "tf_optim_step", "tf_read_adapter",
           "tf_get_steps", "tf_check_status", "tf_profile_enable", "tf_profile_read", "tf_set_lm_backward",
           "tf_set_attention_backward"]

PROJ = ("q", "k", "v", "o", "gate", "up", "down")
HEAD_DIM = 128
TF_PROF_CLASSES = ["routing", "embed", "norm", "shrink", "qkv", "rope", "attn_fwd", "o", "gateup",
                   "down", "lm_fwd", "loss", "lm_dz", "lm_dh", "down_bwd", "gateup_bwd", "o_bwd",
                   "attn_bwd", "qkv_bwd", "grad", "adam", "other"]
_KINDS = {"weight": 0, "grad": 1, "m": 2, "v": 3}


class _TfConfig(ctypes.Structure):
    _fields_ = [("vocab", c_int32), ("d_model", c_int32), ("n_heads", c_int32),
                ("n_kv_heads", c_int32), ("head_dim", c_int32), ("d_ffn", c_int32),
                ("n_layers", c_int32), ("n_adapters", c_int32), ("ranks", POINTER(c_int32)),
                ("alphas", POINTER(c_float)), ("rope_theta", c_float), ("rms_eps", c_float),
                ("max_tokens", c_int64)]


class _TfInit(ctypes.Structure):
    _fields_ = [("E", c_void_p), ("Wout", c_void_p), ("final_norm", c_void_p),
                ("attn_norm", POINTER(c_void_p)), ("mlp_norm", POINTER(c_void_p)),
                ("W", POINTER(c_void_p) * 7), ("A", POINTER(c_void_p) * 7),
                ("B", POINTER(c_void_p) * 7)]


class _TfBatch(ctypes.Structure):
    _fields_ = [("n_tokens", c_int64), ("tokens", c_void_p), ("targets", c_void_p),
                ("positions", c_void_p), ("adapter_ids", c_void_p)]


_SIGNATURES = {
    "mlora_tf_create": (c_int32, [POINTER(_TfConfig), POINTER(_TfInit), POINTER(c_void_p)]),
    "mlora_tf_destroy": (c_int32, [c_void_p]),
    "mlora_tf_forward": (c_int32, [c_void_p, POINTER(_TfBatch), c_void_p, c_void_p]),
    "mlora_tf_forward_backward": (c_int32, [c_void_p, POINTER(_TfBatch), c_int32, POINTER(_LossInputs),
                                            c_void_p, c_void_p, c_void_p]),
    "mlora_tf_forward_backward_custom": (c_int32, [c_void_p, POINTER(_TfBatch), c_void_p, c_void_p,
                                                   c_void_p, c_void_p]),
    "mlora_tf_optim_step": (c_int32, [c_void_p, POINTER(_Adam), POINTER(c_int32), c_int32, c_void_p,
                                      c_void_p]),
    "mlora_tf_read_adapter": (c_int32, [c_void_p, c_int32, c_int32, c_int32, c_int32, c_int32,
                                        c_void_p, c_void_p]),
    "mlora_tf_get_steps": (c_int32, [c_void_p, POINTER(c_int64), c_void_p]),
    "mlora_tf_check_status": (c_int32, [c_void_p, c_void_p]),
    "mlora_tf_profile_enable": (c_int32, [c_void_p, c_int32]),
    "mlora_tf_set_lm_backward": (c_int32, [c_void_p, c_int32]),
    "mlora_tf_set_attention_backward": (c_int32, [c_void_p, c_int32]),
    "mlora_tf_profile_read": (c_int32, [c_void_p, POINTER(c_double), POINTER(c_int64), c_int32]),
    "mlora_tf_kernel_launches": (c_int64, [c_void_p]),
    "mlora_tf_device_bytes": (c_int64, [c_void_p]),
}

_tf_lib = None


def _lib():
    global _tf_lib
    if _tf_lib is None:
        lib = load_library()
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _tf_lib = lib
    return _tf_lib


class TfHandle:
    """Owns one mlora_tf_t*; keeps the shapes it was created with."""

    def __init__(self, ptr: int, n_adapters: int, ranks, d: int, n_heads: int, n_kv_heads: int,
                 f: int, n_layers: int):
        self.ptr = c_void_p(ptr)
        self.n_adapters = n_adapters
        self.ranks = list(ranks)
        self.d, self.f, self.n_layers = d, f, n_layers
        self.n_heads, self.n_kv_heads = n_heads, n_kv_heads

    def shape_of(self, proj: str, factor: str, adapter: int):
        q, kv = self.n_heads * HEAD_DIM, self.n_kv_heads * HEAD_DIM
        out, inp = {"q": (q, self.d), "k": (kv, self.d), "v": (kv, self.d), "o": (self.d, q),
                    "gate": (self.f, self.d), "up": (self.f, self.d), "down": (self.d, self.f)}[proj]
        r = self.ranks[adapter]
        return (r, inp) if factor == "A" else (out, r)

    @property
    def kernel_launches(self) -> int:
        return int(_lib().mlora_tf_kernel_launches(self.ptr))

    @property
    def device_bytes(self) -> int:
        return int(_lib().mlora_tf_device_bytes(self.ptr))

    def __del__(self):
        try:
            if self.ptr and _tf_lib is not None:
                _tf_lib.mlora_tf_destroy(self.ptr)
                self.ptr = c_void_p(0)
        except Exception:  # pragma: no cover - interpreter shutdown
            pass


def tf_create(vocab: int, d_model: int, n_heads: int, n_kv_heads: int, d_ffn: int, n_layers: int,
              ranks: Sequence[int], alphas: Sequence[float], max_tokens: int, base: dict,
              A: Optional[dict] = None, B: Optional[dict] = None, rope_theta: float = 1e6,
              rms_eps: float = 1e-6) -> TfHandle:
    """Create a handle.  base: CUDA bf16 tensors E, Wout, final_norm, lists
    attn_norm[l], mlp_norm[l], and W[p][l] for p in PROJ; A[p][a][l], B[p][a][l]:
    CUDA float32 tensors (or None)."""
    lib = _lib()
    n_ad, L = len(ranks), n_layers
    cfg = _TfConfig(vocab, d_model, n_heads, n_kv_heads, HEAD_DIM, d_ffn, n_layers, n_ad,
                    (c_int32 * n_ad)(*ranks), (c_float * n_ad)(*alphas), rope_theta, rms_eps,
                    max_tokens)
    keep = []

    def arr(ptrs):
        a = (c_void_p * len(ptrs))(*ptrs)
        keep.append(a)
        return ctypes.cast(a, POINTER(c_void_p))

    def table(x):
        if x is None:
            return None
        return arr([x[a][l].data_ptr() if x[a][l] is not None else None
                     for a in range(n_ad) for l in range(L)])

    init = _TfInit()
    init.E, init.Wout, init.final_norm = base["E"].data_ptr(), base["Wout"].data_ptr(), \
        base["final_norm"].data_ptr()
    init.attn_norm = arr([g.data_ptr() for g in base["attn_norm"]])
    init.mlp_norm = arr([g.data_ptr() for g in base["mlp_norm"]])
    for i, p in enumerate(PROJ):
        init.W[i] = arr([w.data_ptr() for w in base["W"][p]])
        init.A[i] = table(A[p]) if A is not None else None
        init.B[i] = table(B[p]) if B is not None else None
    out = c_void_p()
    _check(lib.mlora_tf_create(ctypes.byref(cfg), ctypes.byref(init), ctypes.byref(out)))
    return TfHandle(out.value, n_ad, ranks, d_model, n_heads, n_kv_heads, d_ffn, n_layers)


def tf_destroy(h: TfHandle):
    if h.ptr:
        _check(_lib().mlora_tf_destroy(h.ptr))
        h.ptr = c_void_p(0)


def _batch(tokens, targets, positions, adapter_ids) -> _TfBatch:
    n = int(tokens.numel())
    assert targets.numel() == n and positions.numel() == n and adapter_ids.numel() == n
    return _TfBatch(n, _ptr(tokens), _ptr(targets), _ptr(positions), _ptr(adapter_ids))


def tf_forward(h: TfHandle, tokens, targets, positions, adapter_ids, logprobs_out=None, stream=None):
    import torch
    if logprobs_out is None:
        logprobs_out = torch.empty(tokens.numel(), dtype=torch.float32, device=tokens.device)
    b = _batch(tokens, targets, positions, adapter_ids)
    _check(_lib().mlora_tf_forward(h.ptr, ctypes.byref(b), _ptr(logprobs_out), _stream(stream)))
    return logprobs_out


def tf_forward_backward(h: TfHandle, tokens, targets, positions, adapter_ids, loss_kind: str,
                        weights=None, advantages=None, sampler_logprobs=None, clip_eps: float = 0.2,
                        logprobs_out=None, loss_out=None, stream=None):
    """Returns (logprobs [N] float32, loss per adapter [n_adapters] float64)."""
    import torch
    dev = tokens.device
    if logprobs_out is None:
        logprobs_out = torch.empty(tokens.numel(), dtype=torch.float32, device=dev)
    if loss_out is None:
        loss_out = torch.empty(h.n_adapters, dtype=torch.float64, device=dev)
    b = _batch(tokens, targets, positions, adapter_ids)
    li = _LossInputs(_ptr(weights), _ptr(advantages), _ptr(sampler_logprobs), clip_eps)
    _check(_lib().mlora_tf_forward_backward(h.ptr, ctypes.byref(b), LOSS_KINDS[loss_kind],
                                            ctypes.byref(li), _ptr(logprobs_out), _ptr(loss_out),
                                            _stream(stream)))
    return logprobs_out, loss_out


def tf_forward_backward_custom(h: TfHandle, tokens, targets, positions, adapter_ids, dloss_dlogprobs,
                               logprobs_out=None, loss_out=None, stream=None):
    import torch
    dev = tokens.device
    if logprobs_out is None:
        logprobs_out = torch.empty(tokens.numel(), dtype=torch.float32, device=dev)
    if loss_out is None:
        loss_out = torch.empty(h.n_adapters, dtype=torch.float64, device=dev)
    b = _batch(tokens, targets, positions, adapter_ids)
    _check(_lib().mlora_tf_forward_backward_custom(h.ptr, ctypes.byref(b), _ptr(dloss_dlogprobs),
                                                   _ptr(logprobs_out), _ptr(loss_out), _stream(stream)))
    return logprobs_out, loss_out


def tf_optim_step(h: TfHandle, lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0,
                  adapters: Optional[Sequence[int]] = None, skipped_out=None, stream=None):
    """Adam step; returns the device int32 [n_adapters] skipped flags."""
    import torch
    if skipped_out is None:
        skipped_out = torch.empty(h.n_adapters, dtype=torch.int32, device="cuda")
    p = _Adam(lr, beta1, beta2, eps, weight_decay)
    if adapters is None:
        arr, n = None, 0
    else:
        n = len(adapters)
        arr = (c_int32 * max(1, n))(*adapters)
    _check(_lib().mlora_tf_optim_step(h.ptr, ctypes.byref(p), arr, n, _ptr(skipped_out),
                                      _stream(stream)))
    return skipped_out


def tf_read_adapter(h: TfHandle, adapter: int, layer: int, proj: str, factor: str, kind: str = "weight",
                    stream=None):
    """One fp32 adapter tensor (factor "A" [r x in] or "B" [out x r]) as a CUDA tensor."""
    import torch
    out = torch.empty(h.shape_of(proj, factor, adapter), dtype=torch.float32, device="cuda")
    _check(_lib().mlora_tf_read_adapter(h.ptr, adapter, layer, PROJ.index(proj), 0 if factor == "A" else 1,
                                        _KINDS[kind], _ptr(out), _stream(stream)))
    return out


def tf_get_steps(h: TfHandle, stream=None):
    arr = (c_int64 * h.n_adapters)()
    _check(_lib().mlora_tf_get_steps(h.ptr, arr, _stream(stream)))
    return [int(x) for x in arr]


def tf_check_status(h: TfHandle, stream=None) -> int:
    return int(_lib().mlora_tf_check_status(h.ptr, _stream(stream)))


def tf_set_lm_backward(h: TfHandle, mode: str):
    """LM-head backward mode: "recompute" (default) or "keep_logits"."""
    from . import LM_BACKWARD_MODES
    _check(_lib().mlora_tf_set_lm_backward(h.ptr, LM_BACKWARD_MODES[mode]))


def tf_set_attention_backward(h: TfHandle, max_seq_len: int):
    """0: the query side recomputes S and dP (default); > 0: dS blocks are
    stored for sequences of at most max_seq_len tokens."""
    _check(_lib().mlora_tf_set_attention_backward(h.ptr, int(max_seq_len)))


def tf_profile_enable(h: TfHandle, on: bool = True):
    _check(_lib().mlora_tf_profile_enable(h.ptr, 1 if on else 0))


def tf_profile_read(h: TfHandle, reset: bool = True) -> dict:
    """{class: (milliseconds, launches)} accumulated since the last reset."""
    n = len(TF_PROF_CLASSES)
    ms = (c_double * n)()
    cnt = (c_int64 * n)()
    _check(_lib().mlora_tf_profile_read(h.ptr, ms, cnt, 1 if reset else 0))
    return {TF_PROF_CLASSES[i]: (float(ms[i]), int(cnt[i])) for i in range(n)}
