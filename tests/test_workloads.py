"""The seeded synthetic inputs: a token's activations, routes and route
weights do not depend on how many tokens the layer has (the byte-invariance
tests compare rows across batch sizes on that basis), and every stream is
reproducible."""
import numpy as np

from workloads import MoEWorkload, config


def test_tokens_are_prefixes_of_one_stream():
    for cfg in (1, 3):
        small = MoEWorkload(config(cfg, M=3))
        large = MoEWorkload(config(cfg, M=40))
        assert np.array_equal(small.x, large.x[:3])
        assert np.array_equal(small.ids, large.ids[:3])
        assert np.array_equal(small.rw, large.rw[:3])


def test_expert_weights_are_reproducible_and_independent_of_the_batch():
    a = MoEWorkload(config(0)).projection(3, 1)
    b = MoEWorkload(config(0, M=5)).projection(3, 1)
    assert np.array_equal(a.trellis, b.trellis)
    assert np.array_equal(a.suh, b.suh) and np.array_equal(a.scale, b.scale)
    g = MoEWorkload(config(0)).projection(3, 0)          # gate: same shape as up
    assert g.trellis.shape == a.trellis.shape and not np.array_equal(g.trellis, a.trellis)
