"""The seeded input generators hold the structure the tests and the benchmark rely on (CPU)."""
import math

import numpy as np
import pytest
import torch

from fp8_attention_forward_gb300 import inputs


@pytest.mark.parametrize("kind", ["prefill", "decode"])
def test_lazy_staircase_climbs_half_q_per_tile(kind):
    """Every row's largest log2-unit score rises by exactly 0.5 q per 128 keys, from 0."""
    c = inputs.lazy_staircase(kind)
    q = c.q.float().double()
    k = c.k.float().double()[:, :, 0]  # (B, Sk, D)
    # the E4M3 codes hold the intended values exactly
    assert set(np.unique(q.numpy()).tolist()) <= set(inputs.STAIRCASE_Q_LEVELS)
    assert set(np.unique(k.numpy()).tolist()) <= {0.0, 2.0}
    c_log2 = c.softmax_scale / math.log(2.0)
    for b in range(c.B):
        y = torch.einsum("shd,kd->shk", q[b], k[b]) * c_log2  # (Sq, Hq, Sk)
        tile_max = y.reshape(y.shape[0], y.shape[1], -1, 128).amax(-1)
        qv = q[b, :, :, 0]  # the row's level
        steps = tile_max[..., 1:] - tile_max[..., :-1]
        assert torch.allclose(tile_max[..., 0], torch.zeros_like(qv))
        assert torch.allclose(steps, (0.5 * qv)[..., None].expand_as(steps), atol=1e-12)
    # the rows cycle through every level
    assert set(np.unique(q[..., 0].numpy()).tolist()) == set(inputs.STAIRCASE_Q_LEVELS)


def test_lazy_staircase_kernel_selection_shapes():
    """prefill: 128 packed rows on one kv-head (the 128-row kernel); decode: one-token
    requests with 8 q-heads per kv-head (the decode kernel)."""
    p = inputs.lazy_staircase("prefill")
    d = inputs.lazy_staircase("decode")
    assert p.seqlens_q[0] * (p.Hq // p.Hkv) == 128
    assert d.seqlens_q == [1, 1] and d.Hq // d.Hkv == 8
    assert p.seqlens_k[0] == d.seqlens_k[0] == 64 * 128
