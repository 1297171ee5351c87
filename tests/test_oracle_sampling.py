"""Pins of the oracle's temperature sampling ("Let's make GPT-2 in assembly",
Step 7: divide the scores by a temperature, apply softmax and draw at random;
"gpt2.s" README, Options: -t, 0 means greedy).

The draw is the Gumbel-max form: argmax_i of s_i / T - log(-log u_i).  Its
distribution is pinned against softmax(s / T) computed here in float64, not
against its own formula; the uniform numbers against the uniform law.
"""
import numpy as np
import pytest

from oracle import oracle as orc

scipy_stats = pytest.importorskip("scipy.stats")


def test_uniform_numbers_are_uniform_and_inside_the_open_interval():
    u = np.array([orc.uniform(7, k) for k in range(100_000)])
    assert u.min() > 0.0 and u.max() < 1.0
    assert abs(u.mean() - 0.5) < 0.005
    assert abs(u.var() - 1.0 / 12.0) < 0.002
    counts, _ = np.histogram(u, bins=100, range=(0.0, 1.0))
    assert scipy_stats.chisquare(counts).pvalue > 1e-4
    # neighbouring counters are not correlated
    assert abs(np.corrcoef(u[:-1], u[1:])[0, 1]) < 0.02


def test_uniform_mapping_stays_inside_the_open_interval_at_its_extremes():
    # the largest and smallest raw outputs: the draw must stay below 1 (a
    # draw of exactly 1 gives -log(-log u) = +inf, which would win every
    # argmax) and above 0; the grid is 2^-23 wide, centred in each cell
    top = orc.uniform_bits(2**64 - 1)
    assert top < 1.0 and top == 1.0 - 2.0**-24
    assert orc.uniform_bits(0) == 2.0**-24
    assert orc.uniform_bits(2**41) == 1.5 * 2.0**-23
    # every cell of the top 23 bits maps to a distinct value strictly inside
    for m in (1, 2**22, 2**23 - 2, 2**23 - 1):
        u = orc.uniform_bits(m << 41)
        assert 0.0 < u < 1.0 and u == (m + 0.5) * 2.0**-23


def test_generator_depends_on_seed_and_counter():
    a = [orc.splitmix64(1, k) for k in range(1000)]
    b = [orc.splitmix64(2, k) for k in range(1000)]
    assert len(set(a)) == 1000
    assert sum(x == y for x, y in zip(a, b)) == 0


@pytest.mark.parametrize("temperature", [0.5, 0.8, 1.5])
def test_draws_follow_softmax_of_scores_over_temperature(temperature):
    s = np.array([1.0, 0.5, 0.0, -0.5, 2.0, 0.1, -1.0, 0.3], np.float32)
    n_draws = 40_000
    ids = np.array([orc.sample(s, temperature, 11, pos) for pos in range(n_draws)])
    counts = np.bincount(ids, minlength=s.size)
    z = s.astype(np.float64) / temperature
    p = np.exp(z - z.max())
    p /= p.sum()
    assert scipy_stats.chisquare(counts, p * n_draws).pvalue > 1e-4


def test_temperature_zero_is_greedy_and_tiny_temperature_picks_the_maximum():
    rng = np.random.default_rng(0)
    for _ in range(50):
        s = rng.normal(size=100).astype(np.float32)
        assert orc.sample(s, 0.0, 3, 5) == int(np.argmax(s))
        # Gumbel noise is below ~40 here: 1e-4 * 40 is far below the top-2 gap of these scores
        gap = np.sort(s)[-1] - np.sort(s)[-2]
        if gap > 0.01:
            assert orc.sample(s, 1e-4, 3, 5) == int(np.argmax(s))


def test_very_high_temperature_is_close_to_uniform():
    s = np.array([3.0, -2.0, 0.0, 1.0], np.float32)
    ids = np.array([orc.sample(s, 1e6, 5, pos) for pos in range(20_000)])
    counts = np.bincount(ids, minlength=4)
    assert scipy_stats.chisquare(counts).pvalue > 1e-4


def test_draws_are_reproducible_and_depend_on_position():
    s = np.linspace(-1, 1, 64).astype(np.float32)
    a = [orc.sample(s, 1.0, 9, pos) for pos in range(200)]
    b = [orc.sample(s, 1.0, 9, pos) for pos in range(200)]
    assert a == b
    assert len(set(a)) > 20


def test_scores_are_the_perturbed_logits():
    s = np.array([0.25, -0.75, 1.5], np.float32)
    sc = orc.sample_scores(s, 0.5, 4, 2)
    assert int(np.argmax(sc)) == orc.sample(s, 0.5, 4, 2)
    # the perturbation does not depend on the scores: shifting all scores shifts all perturbed scores alike
    sc2 = orc.sample_scores(s + np.float32(1.0), 0.5, 4, 2)
    assert np.allclose(sc2 - sc, 2.0, atol=1e-5)
