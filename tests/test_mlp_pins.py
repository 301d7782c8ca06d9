"""Pins of the ReLU^2 MLP oracle (one token, batch 1): y = sum over neurons that fired of
h_i w_down_i, h_i = max(w_up_i . x, 0)^2.

Pinned by: weights exactly zero at and below zero and squares above; the rows of dead
neurons never matter (NaN rows there leave y finite and unchanged); one live neuron gives
its own row times h; homogeneity (x -> lambda x scales y by lambda^2); a permutation of the
neurons leaves y unchanged; the generator's live count."""
import numpy as np
import pytest

import gen
import oracle


def _small(seed, d=64, f=96, live=0.25):
    x, wu, wd, mask = gen.make_mlp(seed, d, f, live)
    return (gen.bf16_to_f32(x).astype(np.float64), gen.bf16_to_f32(wu).astype(np.float64),
            gen.bf16_to_f32(wd).astype(np.float64), mask)


def test_weights_are_relu_squared():
    x, wu, wd, _ = _small(1)
    _, h, nl = oracle.relu2_mlp(x, wu, wd)
    a = wu @ x
    assert (h >= 0).all()
    assert np.array_equal(h == 0, a <= 0)
    np.testing.assert_allclose(h[a > 0], a[a > 0] ** 2, rtol=1e-12)
    assert nl == int((a > 0).sum())


@pytest.mark.parametrize("live", [0.0, 0.05, 0.22, 1.0])
def test_live_count_is_the_generators(live):
    x, wu, wd, mask = _small(2, d=128, f=400, live=live)
    _, h, nl = oracle.relu2_mlp(x, wu, wd)
    assert nl == int(mask.sum()) == int(round(live * 400))
    assert np.array_equal(h > 0, mask)


def test_dead_rows_are_never_read():
    x, wu, wd, mask = _small(3)
    y, _, _ = oracle.relu2_mlp(x, wu, wd)
    wd2 = wd.copy()
    wd2[~mask] = np.nan
    y2, _, _ = oracle.relu2_mlp(x, wu, wd2)
    np.testing.assert_array_equal(y, y2)


def test_one_live_neuron():
    rng = np.random.default_rng(4)
    d, f = 32, 10
    x = rng.standard_normal(d)
    wu = -np.tile(x, (f, 1)) * rng.uniform(0.5, 2.0, size=(f, 1))
    wu[6] = 0.3 * x
    wd = rng.standard_normal((f, d))
    y, h, nl = oracle.relu2_mlp(x, wu, wd)
    assert nl == 1
    a = 0.3 * float(x @ x)
    np.testing.assert_allclose(y, a * a * wd[6], rtol=1e-12)


def test_homogeneity_and_permutation():
    x, wu, wd, _ = _small(5)
    y, _, _ = oracle.relu2_mlp(x, wu, wd)
    y2, _, _ = oracle.relu2_mlp(2.0 * x, wu, wd)
    np.testing.assert_allclose(y2, 4.0 * y, rtol=1e-12, atol=1e-12)
    perm = np.random.default_rng(6).permutation(wu.shape[0])
    y3, _, _ = oracle.relu2_mlp(x, wu[perm], wd[perm])
    np.testing.assert_allclose(y3, y, rtol=1e-10, atol=1e-12)
