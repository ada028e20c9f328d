"""The seeded generator: compiled copy equals its numpy restatement; the
workloads have the stated shapes and statistics."""
import numpy as np
import pytest

import inputs
from inputs import CONFIGS, LCE_STRESS, IGNORE_INDEX


def test_c_matches_numpy_restatement():
    for seed, stream, off in [(1234, 5, 0), (42, 0, 17), (7, 99, 1 << 33)]:
        a = inputs.normal(seed, stream, 4097, 0.0, 0.02, offset=off)
        b = inputs.normal_np(seed, stream, 4097, 0.0, 0.02, offset=off)
        assert np.array_equal(a, b)
        assert np.array_equal(inputs.randint(seed, stream, 999, 152064, off),
                              inputs.randint_np(seed, stream, 999, 152064, off))
        assert np.array_equal(inputs.uniform(seed, stream, 333, off),
                              inputs.uniform_np(seed, stream, 333, off))


def test_counter_based_slices():
    full = inputs.normal(1, 2, 1000)
    assert np.array_equal(full[301:777], inputs.normal(1, 2, 476, offset=301))


def test_normal_statistics():
    x = inputs.normal(1234, 3, 1 << 20, 0.0, 0.02).astype(np.float64)
    assert abs(x.mean()) < 1e-4 and abs(x.std() - 0.02) < 1e-4


def test_unit_sizes_match_shapes():
    c = CONFIGS["8b"]
    assert inputs.unit_numel(c, 0) == 218_112_000
    assert inputs.unit_numel(CONFIGS["tiny"], 0) == 791_040
    t = CONFIGS["tiny"]
    assert inputs.unit_numel(t, 0) == 2 * 256 + 3 * 256 * 256 + 256 * 256 + 3 * 256 * 688


def test_tokens_labels_next_token():
    c = CONFIGS["tiny"]
    tok, lab = inputs.tokens_and_labels(c)
    assert tok.shape == (2, 128) and tok.min() >= 0 and tok.max() < c.vocab
    assert np.array_equal(lab[:, :-1], tok[:, 1:]) and (lab[:, -1] == IGNORE_INDEX).all()


def test_lce_inputs_ignore_fraction():
    from inputs.configs import LceConfig
    c = LceConfig("t", 64, 1000, 2, 4096, 0.1)
    h, w, lab = inputs.lce_inputs(c)
    frac = np.mean(lab == IGNORE_INDEX)
    assert 0.09 < frac < 0.11 and lab.max() < 1000
