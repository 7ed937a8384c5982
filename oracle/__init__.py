"""fp64 CPU oracle for Hedgehog / Taylor causal linear attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call,
link or execute this package: only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` use it.  It shares no code with the CUDA
path (``softmax_mimicking_feature_gb300``) and imports nothing from it.

Every function is a plain, definition-level restatement of the method in
float64 with numpy; library primitives used as single steps are ``@``
(matrix product), ``exp``, ``log`` and sums.  No blocking, chunking or fusion
is done here beyond what the definition states.

Pinned by ``tests/test_oracle_pins.py`` (closed forms, invariants, hand-worked
tiny cases).  Every function has at least one pin; none is "parity unpinned".
"""

from .hedgehog_oracle import (  # noqa: F401
    hedgehog_feature_map,
    hedgehog_softmax_feature_map,
    taylor2_feature_map,
    taylor2_feature_dim,
    feature_map,
    causal_weights,
    linattn_quadratic,
    linattn_rows,
    linattn_recurrent,
    decode_step,
    softmax_target,
    mimicry_loss,
    mimicry_loss_rows,
    fwd_causal,
    mimicry_loss_grad,
    loss_grad_causal,
    attention_entropy,
    mimicry_stats,
    stats_causal,
    loss_causal,
)
