"""CPU oracle for the Llama decoder forward pass — TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct numpy restatement of what the CUDA path
computes, written from the pages' description of the method and checked
against closed forms, invariants and brute force (``tests/test_oracle_*.py``).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package.  The product path (the C-ABI
library and its Python binding) never imports, calls or links it, and it
shares no code with that path: the only module both sides use is ``synth``,
which draws seeded inputs and holds none of the method's arithmetic.

Every function in ``oracle.llama`` is pinned by at least one test that does
not restate its formula; none is "parity unpinned".
"""
from .llama import (  # noqa: F401
    Hparams, Model, Context, bf16_to_float, rms_norm, rope_angles, rope,
    attention_one_seq, silu, swiglu_mlp, layer_forward, forward_ubatch,
    greedy_argmax, generate_greedy, OK, NO_KV_ROOM, INVALID,
)
