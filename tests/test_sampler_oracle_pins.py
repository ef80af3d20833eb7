"""Pins of the sampler-chain oracle (oracle/sampler.py) to what the article and the mathematics fix,
independently of the oracle's own code: hand-computed penalty values, argmax, the softmax closed
form (the frequency of each token over a uniform grid of random numbers equals its probability),
hand-built distributions for top-k / top-p / min-p, ties and the order of the chain."""
import math

import numpy as np
import pytest

from oracle import sampler as S

GRID = 4000   # random numbers u_j = (j + 1/2) / GRID


def freqs(logits, **kw):
    """Fraction of the u grid that the chain maps to each token."""
    V = len(logits)
    cnt = np.zeros(V)
    for j in range(GRID):
        cnt[S.sample_chain(np.asarray(logits, np.float32), u=(j + 0.5) / GRID, **kw)] += 1
    return cnt / GRID


def softmax(x):
    x = np.asarray(x, np.float64)
    e = np.exp(x - x.max())
    return e / e.sum()


def test_penalty_hand_values():
    # 2.0 / 1.5 = 4/3 rounded to float32; -1.0 * 1.5 = -1.5; duplicates count once; -1 and 4 ignored
    got = S.penalize(np.array([2.0, 1.9, -1.0, -1.2], np.float32), [0, 2, 0, -1, 4], 1.5)
    assert got.dtype == np.float32
    assert got[0] == np.float32(4.0 / 3.0) and got[2] == np.float32(-1.5)
    assert got[1] == np.float32(1.9) and got[3] == np.float32(-1.2)
    # the penalty moves the greedy choice from token 0 to token 1
    assert S.sample_chain(np.array([2.0, 1.9], np.float32), [0], 1.5, temp=0.0) == 1
    # a negative logit is pushed further down: -1 * 1.5 = -1.5 < -1.2
    assert S.sample_chain(np.array([-1.0, -1.2], np.float32), [0], 1.5, temp=0.0) == 1


def test_greedy_is_argmax_lowest_index_on_ties():
    rng = np.random.default_rng(7)
    for _ in range(20):
        x = rng.integers(-3, 4, size=50).astype(np.float32)   # many ties
        assert S.sample_chain(x, temp=0.0) == int(np.argmax(x))
        assert S.sample_chain(x, top_k=1, temp=0.7, u=0.99) == int(np.argmax(x))
    assert S.sample_chain(np.array([0.0, -0.0, -1.0], np.float32), temp=0.0) == 0
    assert S.sample_chain(np.array([-0.0, 0.0, -1.0], np.float32), temp=0.0) == 0


def test_draw_matches_softmax():
    logits = np.array([0.3, -1.2, 2.0, 0.0, 1.1, -0.4, 0.9, -2.5], np.float32)
    for T in (1.0, 0.5, 2.0):
        f = freqs(logits, temp=T)
        p = softmax(logits.astype(np.float64) / T)
        assert np.all(np.abs(f - p) <= 1.0 / GRID + 1e-12), (T, f, p)


def test_temperature_two_tokens_closed_form():
    logits = np.array([0.0, math.log(3.0)], np.float32)
    assert abs(freqs(logits, temp=1.0)[0] - 0.25) <= 1.0 / GRID
    assert abs(freqs(logits, temp=2.0)[0] - 1.0 / (1.0 + math.sqrt(3.0))) <= 1.0 / GRID


def test_top_p_hand_distribution():
    probs = np.array([0.05, 0.5, 0.15, 0.3])          # leader id 1, then 3, 2, 0
    logits = np.log(probs).astype(np.float32)
    assert set(np.nonzero(freqs(logits, top_p=0.45))[0]) == {1}
    f = freqs(logits, top_p=0.79)                      # 0.5 < 0.79 <= 0.8
    assert set(np.nonzero(f)[0]) == {1, 3}
    assert abs(f[1] - 0.5 / 0.8) <= 1.0 / GRID + 1e-6
    assert set(np.nonzero(freqs(logits, top_p=0.81))[0]) == {1, 2, 3}


def test_min_p_hand_distribution():
    probs = np.array([0.05, 0.5, 0.15, 0.3])
    logits = np.log(probs).astype(np.float32)
    assert set(np.nonzero(freqs(logits, min_p=0.5))[0]) == {1, 3}        # p >= 0.25
    assert set(np.nonzero(freqs(logits, min_p=0.2))[0]) == {1, 2, 3}     # p >= 0.10
    assert set(np.nonzero(freqs(logits, min_p=0.05))[0]) == {0, 1, 2, 3}
    assert set(np.nonzero(freqs(logits, min_p=5.0))[0]) == {1}           # at least the leader


def test_top_k_ties_keep_lower_ids():
    f = freqs(np.array([1.0, 1.0, 1.0, 0.0], np.float32), top_k=2)
    assert set(np.nonzero(f)[0]) == {0, 1}
    assert abs(f[0] - 0.5) <= 1.0 / GRID


def test_top_p_renormalises_over_top_k_survivors():
    # over the 2 survivors of top-k the leader holds 0.5 / 0.8 = 0.625 >= 0.6: only it remains;
    # over the whole row it would hold 0.5 < 0.6 and top-p alone keeps two tokens
    logits = np.log(np.array([0.5, 0.3, 0.2])).astype(np.float32)
    assert set(np.nonzero(freqs(logits, top_k=2, top_p=0.6))[0]) == {0}
    assert set(np.nonzero(freqs(logits, top_p=0.6))[0]) == {0, 1}


def test_draw_walks_ids_upwards():
    # equal weights: u just below 1/3 picks the lowest id, just above 2/3 the highest
    logits = np.zeros(3, np.float32)
    assert S.sample_chain(logits, u=0.33) == 0
    assert S.sample_chain(logits, u=0.34) == 1
    assert S.sample_chain(logits, u=0.67) == 2
    assert S.sample_chain(logits, u=0.0) == 0


@pytest.mark.parametrize("seed", [0, 1])
def test_acceptable_set_is_one_token_away_from_boundaries(seed):
    rng = np.random.default_rng(seed)
    x = rng.normal(0, 2, 1000).astype(np.float32)
    s = S.acceptable_tokens(x, top_k=50, top_p=0.9, min_p=0.05, temp=0.8, u=0.37)
    assert S.sample_chain(x, top_k=50, top_p=0.9, min_p=0.05, temp=0.8, u=0.37) in s
    assert 1 <= len(s) <= 2
