"""The seeded input recipe: deterministic draws, the stated distributions,
and the skew of the DeepSeek-V3-shaped router logits (a fixed 20% of the
experts receive about half of the (token, slot) assignments)."""
import numpy as np

from int4_group_quantized_int4g_gb300 import inputs
from oracle import int4g_oracle as O


def test_draws_are_deterministic_and_streams_differ():
    a = inputs.dense_weight(64, 256, layer=3)
    b = inputs.dense_weight(64, 256, layer=3)
    c = inputs.dense_weight(64, 256, layer=4)
    assert np.array_equal(a, b) and not np.array_equal(a, c)
    assert np.array_equal(inputs.activations(4, 256, stream=1), inputs.activations(4, 256, stream=1))
    assert not np.array_equal(inputs.activations(4, 256, stream=1), inputs.activations(4, 256, stream=2))


def test_dense_weight_outliers():
    """round(0.1% N K) entries multiplied by 20, the rest ~N(0, 0.02)."""
    N, K = 256, 1024
    W = inputs.dense_weight(N, K, layer=7)
    base = inputs.dense_weight(N, K, layer=7, outliers=False)
    changed = np.nonzero((W != base).reshape(-1))[0]
    assert changed.size == round(0.001 * N * K)
    assert np.allclose(W.reshape(-1)[changed], 20 * base.reshape(-1)[changed], rtol=1e-6)
    assert abs(base.std() - 0.02) < 0.001


def test_activations_are_bf16_of_standard_normal():
    x = O.bf16_value(inputs.activations(64, 1024, stream=5))
    assert abs(x.mean()) < 0.02 and abs(x.std() - 1.0) < 0.02
    # bf16 values: at most 8 significant bits
    m, _ = np.frexp(x[x != 0])
    assert np.all(m * 256 == np.round(m * 256))


def test_deepseek_router_skew():
    """256 experts, top-8 of sigmoid scores; the 51 hot experts (+0.67 on
    their N(0,1) logits) take about half of the assignments at M=1024."""
    M, E, k = 1024, 256, 8
    logits = inputs.router_logits(M, E, stream=1024, hot=51)
    hot = inputs.hot_experts(E, 51)
    assert hot.size == 51 and np.unique(hot).size == 51
    ids, _ = O.route(logits, k, O.SIGMOID, True)
    share = np.isin(ids, hot).mean()
    assert 0.45 <= share <= 0.55, share
