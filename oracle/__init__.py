"""CPU fp64 oracle of the multi-tenant LoRA training step.

TEST INFRASTRUCTURE: importable only by tests/, ``__graft_entry__.smoke()``
and the benchmark's CPU-baseline leg.  It shares no code with the CUDA
library and never calls it.
"""
from .mlora_oracle import (LOSS_KINDS, TENSORS, TILE_M, Oracle, adam_update,  # noqa: F401
                           logsumexp_rows, read_state_file, routing, silu,
                           silu_grad, token_loss, write_state_file, load_state_file)
from .transformer_oracle import PROJ, TransformerOracle  # noqa: F401
