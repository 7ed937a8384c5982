"""Why the bias gradient of bf16 inputs has its own tolerance.

The bias gradient db = sum_t dL/dh_t sums over every query and key row and
cancels heavily, so the rounding of the features phi(q), phi(k) to bf16 (the
operand precision of the tensor-core path) moves it more than it moves dW or
any forward output.  This test measures that effect with the fp64 oracle
alone: the same chain rule ("The Attention Weight Distillation Loss"; the map
of "The Hedgehog MLP Feature Map", Choices 1 and 3) evaluated once exactly and
once with only the features rounded to bf16.  On the seeded inputs of the GPU
test with 14 query heads sharing 2 key/value heads (the largest case), that
rounding alone moves db by more than the 5e-3 forward bound and by less than
DB_TOL_BF16, while dW stays inside 5e-3.  Any kernel whose features are bf16
therefore cannot be held to 5e-3 on db, and 1e-2 leaves it the same room
again for its own rounding.  No GPU is involved."""

import numpy as np
import torch

import oracle as O
from softmax_mimicking_feature_gb300 import workloads as wl
from tests._util import BF16_TOL, DB_TOL_BF16, rel_l2_per_head


def _bf16(a):
    """Round-to-nearest-even to bf16, returned in float64."""
    return torch.from_numpy(np.ascontiguousarray(a)).to(torch.float32).to(
        torch.bfloat16).to(torch.float64).numpy()


def _gqa_inputs(seed=37):
    # the GPU test's case: GPT-2 shape, 14 query heads, 2 key/value heads,
    # n = 300; query head h reads key/value head h // 7
    w = wl.WORKLOADS["gpt2_prefill_8x12x1024_d64"].with_(B=1, H=14, n=300)
    x = wl.make_inputs(w, seed=seed)
    q = x["q"].double().numpy()
    k = x["k"][:, :2].double().numpy()
    k = np.repeat(k, 7, axis=1)
    return q, k, x["W"].double().numpy(), x["b"].double().numpy()


def test_bf16_features_alone_move_db_beyond_the_forward_bound():
    q, k, W, b = _gqa_inputs()
    exact = O.loss_grad_causal(q, k, W, b)
    rounded = O.loss_grad_causal(q, k, W, b, feature_rounding=_bf16)
    err_dW = rel_l2_per_head(rounded[0], exact[0], lead=1)
    err_db = rel_l2_per_head(rounded[1], exact[1], lead=1)
    assert err_dW <= BF16_TOL, err_dW
    assert BF16_TOL < err_db < DB_TOL_BF16, err_db


def test_feature_rounding_hook_is_inert_when_exact():
    # the hook only rounds: the identity leaves the gradient bit for bit
    q, k, W, b = _gqa_inputs()
    q, k = q[:, :2, :40], k[:, :2, :40]
    W, b = W[:2], b[:2]
    a = O.loss_grad_causal(q, k, W, b)
    c = O.loss_grad_causal(q, k, W, b, feature_rounding=lambda t: t)
    for x, y in zip(a, c):
        if x is None:
            assert y is None
        else:
            assert np.array_equal(x, y)
