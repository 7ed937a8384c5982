"""Hedgehog / Taylor causal linear attention for GB300 (sm_103a).

The compute path is the C-ABI library ``_lib/libhh.so`` (include/hh.h);
``api`` is its PyTorch binding.  ``workloads`` draws seeded synthetic inputs.
"""

from .api import (  # noqa: F401
    FeatureMap,
    HHError,
    feature_map,
    fmap_dim,
    fwd_plan,
    fwd_workspace_bytes,
    linattn_decode_step,
    linattn_fwd_causal,
    linattn_fwd_causal_from_state,
    fwd_from_state_workspace_bytes,
    loss_workspace_bytes,
    loss_grad_workspace_bytes,
    mimicry_loss,
    mimicry_loss_grad,
    mimicry_stats,
)
