"""CPU pins of the fixed-order lambda the GPU partition tests hand the
oracle (the mean curvature of GraceKV "01 Curvature-guided partition")."""
import math

import numpy as np

from tests.partition_lambda import partition_lambda


def test_equals_the_mean_to_rounding():
    rng = np.random.default_rng(5)
    for end in (16, 511, 512, 513, 4097, 32640):
        k = rng.random(end).astype(np.float32).astype(np.float64) * 2.0
        lam = partition_lambda(k, end)
        assert abs(lam - math.fsum(k) / end) <= 1e-14 * abs(lam)


def test_exact_when_every_sum_is_representable():
    # multiples of 2^-10 below 2: every partial sum is exact in float64
    rng = np.random.default_rng(6)
    end = 3000
    k = rng.integers(0, 2048, end) / 1024.0
    assert partition_lambda(k, end) == sum(k.tolist()) / end


def test_only_the_first_end_values_count():
    k = np.r_[np.ones(100), np.full(50, 7.0)]
    assert partition_lambda(k, 100) == 1.0
