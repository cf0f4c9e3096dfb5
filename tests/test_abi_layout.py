"""The Python binding and the C headers agree (CPU only, no GPU).

A C program compiled with the host compiler against include/mlora.h and
include/mlora_tf.h prints the size and field offsets of every struct the
binding mirrors with ctypes, and the values of the enums and limits it
repeats; the binding's ctypes layouts and constants must match them.  Each
entry point the binding declares must exist in a header with the same
number of parameters and a return type of the same width.
"""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (C struct, ctypes class path, fields in declaration order)
STRUCTS = [
    ("mlora_config", "rl_step_gb300._Config",
     ["vocab", "d_model", "d_ffn", "n_layers", "dtype", "n_adapters", "ranks", "alphas",
      "max_tokens"]),
    ("mlora_init", "rl_step_gb300._Init", ["E", "W1", "W2", "Wout", "A1", "B1", "A2", "B2"]),
    ("mlora_batch", "rl_step_gb300._Batch", ["n_tokens", "tokens", "targets", "adapter_ids"]),
    ("mlora_loss_inputs", "rl_step_gb300._LossInputs",
     ["weights", "advantages", "sampler_logprobs", "clip_eps"]),
    ("mlora_adam", "rl_step_gb300._Adam", ["lr", "beta1", "beta2", "eps", "weight_decay"]),
    ("mlora_tf_config", "rl_step_gb300.transformer._TfConfig",
     ["vocab", "d_model", "n_heads", "n_kv_heads", "head_dim", "d_ffn", "n_layers", "n_adapters",
      "ranks", "alphas", "rope_theta", "rms_eps", "max_tokens"]),
    ("mlora_tf_init", "rl_step_gb300.transformer._TfInit",
     ["E", "Wout", "final_norm", "attn_norm", "mlp_norm", "W", "A", "B"]),
    ("mlora_tf_batch", "rl_step_gb300.transformer._TfBatch",
     ["n_tokens", "tokens", "targets", "positions", "adapter_ids"]),
]

CONSTANTS = ["MLORA_TILE_M", "MLORA_MAX_RANK", "MLORA_CROSS_ENTROPY", "MLORA_IMPORTANCE_SAMPLING",
             "MLORA_PPO", "MLORA_BF16", "MLORA_FP32", "MLORA_A1", "MLORA_B2", "MLORA_GRAD_A1",
             "MLORA_V_B2", "MLORA_TF_HEAD_DIM", "MLORA_TF_NPROJ", "MLORA_NOALLOC_MAX_TOKENS",
             "MLORA_NOALLOC_MAX_ADAPTERS", "MLORA_E_ARG", "MLORA_E_RANGE", "MLORA_E_CUDA",
             "MLORA_E_NOMEM", "MLORA_E_TIMEOUT", "MLORA_E_IO", "MLORA_E_UNSUPPORTED",
             "MLORA_LM_RECOMPUTE", "MLORA_LM_KEEP_LOGITS"]


def _resolve(path):
    import importlib
    mod, name = path.rsplit(".", 1)
    return getattr(importlib.import_module(mod), name)


@pytest.fixture(scope="module")
def c_layout(tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no host C compiler")
    lines = ['#include <stdio.h>', '#include "mlora_tf.h"', "int main(void) {"]
    for cname, _, fields in STRUCTS:
        lines.append(f'  printf("size {cname} %zu\\n", sizeof({cname}));')
        for f in fields:
            lines.append(f'  printf("off {cname}.{f} %zu\\n", offsetof({cname}, {f}));')
    for k in CONSTANTS:
        lines.append(f'  printf("const {k} %lld\\n", (long long)({k}));')
    lines += ["  return 0;", "}"]
    d = tmp_path_factory.mktemp("abi")
    src, exe = d / "layout.c", d / "layout"
    src.write_text("\n".join(lines) + "\n")
    subprocess.run([cc, "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe)], check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    res = {}
    for ln in out.splitlines():
        kind, key, val = ln.split()
        res[(kind, key)] = int(val)
    return res


@pytest.mark.parametrize("cname,cls,fields", STRUCTS, ids=[s[0] for s in STRUCTS])
def test_ctypes_struct_matches_the_header(c_layout, cname, cls, fields):
    S = _resolve(cls)
    assert [f[0] for f in S._fields_] == fields
    assert ctypes.sizeof(S) == c_layout[("size", cname)]
    for f in fields:
        assert getattr(S, f).offset == c_layout[("off", f"{cname}.{f}")], f


def test_binding_constants_match_the_header(c_layout):
    import rl_step_gb300 as m
    import rl_step_gb300.transformer as t
    c = {k: c_layout[("const", k)] for k in CONSTANTS}
    assert m.TILE_M == c["MLORA_TILE_M"] and m.MAX_RANK == c["MLORA_MAX_RANK"]
    assert m.LOSS_KINDS == {"cross_entropy": c["MLORA_CROSS_ENTROPY"],
                            "importance_sampling": c["MLORA_IMPORTANCE_SAMPLING"],
                            "ppo": c["MLORA_PPO"]}
    assert m.LM_BACKWARD_MODES == {"recompute": c["MLORA_LM_RECOMPUTE"],
                                   "keep_logits": c["MLORA_LM_KEEP_LOGITS"]}
    assert m.TENSOR_IDS["A1"] == c["MLORA_A1"] and m.TENSOR_IDS["B2"] == c["MLORA_B2"]
    assert m.TENSOR_IDS["gA1"] == c["MLORA_GRAD_A1"] and m.TENSOR_IDS["vB2"] == c["MLORA_V_B2"]
    assert t.HEAD_DIM == c["MLORA_TF_HEAD_DIM"] and len(t.PROJ) == c["MLORA_TF_NPROJ"]
    codes = {"E_ARG": "MLORA_E_ARG", "E_RANGE": "MLORA_E_RANGE", "E_CUDA": "MLORA_E_CUDA",
             "E_NOMEM": "MLORA_E_NOMEM", "E_TIMEOUT": "MLORA_E_TIMEOUT", "E_IO": "MLORA_E_IO",
             "E_UNSUPPORTED": "MLORA_E_UNSUPPORTED"}
    assert {v: k for k, v in m._ERRORS.items()} == {k: c[v] for k, v in codes.items()}


def _declarations():
    """name -> (return type, parameter count) of every mlora_* function in include/*.h."""
    decls = {}
    for hdr in ("mlora.h", "mlora_tf.h"):
        src = open(os.path.join(ROOT, "include", hdr)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for mt in re.finditer(r"^\s*((?:const\s+)?[\w]+\s*\**)\s*(mlora_\w+)\s*\(([^)]*)\)\s*;",
                              src, flags=re.M):
            ret, name, params = mt.group(1).replace(" ", ""), mt.group(2), mt.group(3).strip()
            n = 0 if params in ("", "void") else len(params.split(","))
            decls[name] = (ret, n)
    return decls


def test_binding_signatures_match_the_header():
    import rl_step_gb300 as m
    import rl_step_gb300.transformer as t
    decls = _declarations()
    width = {"int": ctypes.c_int32, "int64_t": ctypes.c_int64, "constchar*": ctypes.c_char_p}
    sigs = dict(m._SIGNATURES)
    sigs.update(t._SIGNATURES)
    for name, (res, args) in sigs.items():
        assert name in decls, f"{name} is not declared in include/*.h"
        ret, n = decls[name]
        assert len(args) == n, f"{name}: binding passes {len(args)} arguments, header has {n}"
        assert ctypes.sizeof(res) == ctypes.sizeof(width[ret]), name
