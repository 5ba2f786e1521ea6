"""Pins for the exponential-race sampler oracle (CPU only)."""

import math

import numpy as np
import pytest

import oracle


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


def test_philox_known_answer(orc):
    """Philox4x32-10 of the zero counter under the zero key, the generator's
    published known answer."""
    assert orc.philox4x32_10([0, 0, 0, 0], [0, 0]) == [0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8]


def test_uniforms_are_uniform_and_distinct(orc):
    u = np.array([orc.uniform(3, i, 1234, 7) for i in range(20000)])
    assert (u > 0).all() and (u < 1).all()
    assert abs(u.mean() - 0.5) < 0.01 and abs(u.var() - 1 / 12) < 0.005
    assert len(set(u.tolist())) > 19900
    assert orc.uniform(3, 5, 1234, 7) != orc.uniform(4, 5, 1234, 7) != orc.uniform(3, 5, 1234, 8)


def test_race_samples_the_softmax_distribution(orc):
    """The winner of the race is distributed as softmax(logits / T): a
    chi-square test over 60000 independent rows (p-value > 1e-4)."""
    from scipy.stats import chisquare
    V, B, T = 8, 60000, 0.7
    base = np.array([1.0, 0.5, -0.3, 2.0, 0.0, -1.0, 1.5, 0.2], np.float32)
    logits = np.tile(base, (B, 1))
    tok = orc.sample(logits, np.full(B, T, np.float32), seed=99, offset=0)
    z = base.astype(np.float64) / T
    p = np.exp(z - z.max())
    p /= p.sum()
    counts = np.bincount(tok, minlength=V)
    assert chisquare(counts, p * counts.sum()).pvalue > 1e-4


def test_dominant_logit_always_wins(orc):
    logits = np.zeros((50, 1000), np.float32)
    logits[:, 417] = 100.0
    tok = orc.sample(logits, np.ones(50, np.float32), seed=1, offset=0)
    assert (tok == 417).all()


def test_low_temperature_approaches_argmax_and_bad_temperature(orc):
    rng = np.random.default_rng(0)
    logits = rng.standard_normal((40, 500)).astype(np.float32)
    tok = orc.sample(logits, np.full(40, 1e-3, np.float32), seed=5, offset=3)
    assert (tok == logits.argmax(axis=1)).all()
    bad = orc.sample(logits[:3], np.array([0.0, -1.0, math.inf], np.float32), seed=5)
    assert (bad == -1).all()


def test_scores_agree_with_tokens(orc):
    rng = np.random.default_rng(1)
    logits = rng.standard_normal((20, 300)).astype(np.float32)
    tok, sc = orc.sample(logits, np.full(20, 0.9, np.float32), seed=8, offset=0, with_scores=True)
    assert (sc.argmax(axis=1) == tok).all()
