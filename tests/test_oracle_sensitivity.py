"""Pins of the layer-sensitivity oracle (FastJEV Eq. 5-6)."""
import math

import numpy as np

from oracle import sensitivity as sens


def test_hand_example():
    z = np.array([1.0, 2.0, 3.0])                 # ctr = (-1, 0, 1), rms = sqrt(2/3)
    z_skip = np.array([[1.0, 2.0, 4.0],           # delta = (0, 0, 1): ctr = (-1/3, -1/3, 2/3), rms = sqrt(2)/3
                       [5.0, 6.0, 7.0]])          # a common shift only: d = 0
    d, J, sel = sens.layer_sensitivity(z, z_skip, [0, 3], 1)
    assert abs(d[0, 0] - (math.sqrt(2) / 3) / math.sqrt(2 / 3)) < 1e-15
    assert abs(d[1, 0]) < 1e-15
    assert list(sel) == [1]


def test_invariances():
    rng = np.random.default_rng(0)
    z = rng.normal(size=7)
    dz = rng.normal(size=(3, 7))
    d0, _, _ = sens.layer_sensitivity(z, z + dz, [0, 7], 1)
    d1, _, _ = sens.layer_sensitivity(z + 4.0, z + 4.0 + dz + 2.5, [0, 7], 1)    # shifts cancel
    np.testing.assert_allclose(d1, d0, rtol=1e-12)
    d2, _, _ = sens.layer_sensitivity(3 * z, 3 * z + dz, [0, 7], 1)              # scale of z divides d
    np.testing.assert_allclose(d2, d0 / 3, rtol=1e-12)


def test_epsilon_floor_and_mean_over_inputs():
    z = np.array([2.0, 2.0, 1.0, 3.0])              # input 0 constant (rms 0), input 1 = (1, 3)
    z_skip = np.array([[2.0, 2.5, 1.0, 3.0]])
    d, J, _ = sens.layer_sensitivity(z, z_skip, [0, 2, 4], 1)
    assert abs(d[0, 0] - 0.25 / 1e-8) < 1e-3        # rms(ctr((0, 0.5))) = 0.25 over the eps floor
    assert d[0, 1] == 0.0
    assert J[0] == (d[0, 0] + d[0, 1]) / 2


def test_ties_resolved_by_layer_index():
    z = np.array([0.0, 1.0])
    z_skip = np.array([[0.0, 2.0], [0.0, 0.0], [0.0, 2.0], [0.0, 1.0]])   # J = 1, 1, 1, 0
    _, J, sel = sens.layer_sensitivity(z, z_skip, [0, 2], 3)
    assert list(sel) == [3, 0, 1]
