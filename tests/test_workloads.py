"""Input recipe checks (CPU): shapes, dtypes, seeding, and the skewed-load bias."""

import math

import numpy as np
import torch

from oracle import moe_oracle as O
from routing_dispatch_expert_04_b300.workloads import WORKLOADS, ZIPF_BETA, ZIPF_S, make_inputs


def test_tiny_shapes_and_seed():
    wl = WORKLOADS["tiny"]
    a = make_inputs(wl, "cpu", seed=0)
    b = make_inputs(wl, "cpu", seed=0)
    assert a["x"].shape == (256, 128) and a["x"].dtype == torch.float32
    assert a["w_r"].shape == (8, 128)
    assert a["w1"].shape == (8, 512, 128) and a["w2"].shape == (8, 128, 512)
    assert a["b_r"] is None
    for k in ("x", "w_r", "w1", "w2"):
        assert torch.equal(a[k], b[k])
    # N(0, 1/fan_in): sample standard deviations within a few percent
    assert abs(a["w1"].std().item() * math.sqrt(128) - 1) < 0.02
    assert abs(a["w2"].std().item() * math.sqrt(512) - 1) < 0.02


def test_bf16_cast_and_bias_kinds():
    wl = WORKLOADS["dsv3"].scaled(16)
    a = make_inputs(wl, "cpu", weights=False)
    assert a["x"].dtype == torch.bfloat16 and a["b_r"].dtype == torch.float32
    assert a["b_r"].shape == (256,)
    wl = WORKLOADS["long"].scaled(16)
    a = make_inputs(wl, "cpu", weights=False)
    b = a["b_r"].numpy()
    assert b.max() == 0.0                       # rank 1 has zero bias
    ranks = np.sort(np.exp(-b / (ZIPF_BETA * ZIPF_S)))
    assert np.allclose(ranks, np.arange(1, 9), rtol=1e-5)


def test_zipf_bias_gives_forty_percent_top_share():
    """Under i.i.d. N(0,1) logit noise, top-2 routing with the Zipf bias sends ~40% of the
    assignments to the rank-1 expert (the stated recipe of the 64K-token workload)."""
    rng = np.random.default_rng(123)
    E = 8
    bias = -ZIPF_BETA * ZIPF_S * np.log(np.arange(1, E + 1))
    L = (rng.standard_normal((200000, E)) + bias).astype(np.float32)
    ids = O.top_k(L, 2)
    share = (ids == 0).sum() / ids.size
    assert abs(share - 0.40) < 0.01
