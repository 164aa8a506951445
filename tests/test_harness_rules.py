"""The GPU acceptance rule for draft tokens (tests/harness.py), on its own:
a draft may differ from the oracle's argmax only at near-ties."""
import numpy as np
import pytest

from tests import harness as H


def _row(top, second):
    lg = np.zeros((1, 5))
    lg[0, 1], lg[0, 3] = top, second
    return lg


def test_exact_argmax_passes():
    assert H.assert_drafts_match(np.array([1]), _row(4.2, 4.0)) == 0


def test_small_oracle_margin_excuses_a_flip():
    assert H.assert_drafts_match(np.array([3]), _row(4.19, 4.185)) == 1   # margin 0.005 < 1e-2


def test_a_flip_explained_by_the_gpu_logit_errors_passes():
    lg = _row(4.19267, 4.18088)            # margin 0.0118
    gl = lg.copy()
    gl[0, 1], gl[0, 3] = 4.18350, 4.18643  # errors 0.0092 and 0.0055, GPU ranks token 3 first
    assert H.assert_drafts_match(np.array([3]), lg, gpu_logits=gl) == 1


def test_a_flip_without_gpu_logits_fails():
    with pytest.raises(AssertionError):
        H.assert_drafts_match(np.array([3]), _row(4.19267, 4.18088))


def test_a_flip_the_gpu_errors_do_not_explain_fails():
    lg = _row(4.19267, 4.18088)
    with pytest.raises(AssertionError):   # GPU logits equal the oracle's
        H.assert_drafts_match(np.array([3]), lg, gpu_logits=lg.copy())


def test_a_flip_against_the_gpus_own_ranking_fails():
    lg = _row(4.19267, 4.18088)
    gl = lg.copy()
    gl[0, 1], gl[0, 3] = 4.20, 4.17        # large errors, but the GPU itself ranks token 1 first
    with pytest.raises(AssertionError):
        H.assert_drafts_match(np.array([3]), lg, gpu_logits=gl)


def test_errors_beyond_the_per_logit_bound_fail():
    lg = _row(1.0, 0.0)                    # margin 1.0; row RMS ~0.45, bound ~0.022
    gl = lg.copy()
    gl[0, 1], gl[0, 3] = 0.4, 0.6
    with pytest.raises(AssertionError):
        H.assert_drafts_match(np.array([3]), lg, gpu_logits=gl)
