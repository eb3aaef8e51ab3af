"""The seeded input generators: reproducible, and each activation structure is what its
docstring says (these inputs drive the parity tests of the block-scaled M = 1 kernel)."""
import numpy as np
import pytest

import synth
from oracle import numerics


def draw(kind, M=4, K=1024, seed=5):
    return synth.activation_variant(synth.generator(seed, M, K), M, K, kind)


@pytest.mark.parametrize("kind", synth.ACTIVATION_KINDS)
def test_activation_variant_reproducible_and_finite(kind):
    a, b = draw(kind), draw(kind)
    assert a.dtype == np.uint16 and a.shape == (4, 1024)
    assert np.array_equal(a, b)
    assert np.isfinite(numerics.bf16_to_f64(a)).all()


def test_activation_variant_structures():
    v = {k: np.abs(numerics.bf16_to_f64(draw(k))) for k in synth.ACTIVATION_KINDS}
    assert not v["zero"].any()
    assert 0.05 < np.mean(v["sparse"] > 0) < 0.15
    assert 2.0 ** -95 < v["tiny"].max() < 2.0 ** -85
    assert 2.0 ** 85 < v["huge"].max() < 2.0 ** 95
    # outlier channels are the same in every row and about 1000 times the rest
    col = v["outlier"].max(axis=0)
    assert col.max() > 100 * np.median(col)
    # per-run scales differ by many binades within a row
    runs = v["mixed_scale"].reshape(4, -1, 64).max(axis=2)
    assert (np.log2(runs.max(axis=1) / runs.min(axis=1)) > 20).all()
