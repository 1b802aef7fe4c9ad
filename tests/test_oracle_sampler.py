"""Pins of the Gumbel-max sampler oracle against what the sampler page and
the mathematics fix ([NV12 §12.2 "采样器"]), CPU only.

* With every draw equal, dividing by it changes nothing: the sample is the
  greedy argmax of the logits (first maximum).
* With equal logits the softmax is uniform: the sample is the smallest draw.
* The Gumbel-max theorem (the page's derivation): over many independent
  draws the sample frequencies are softmax(logits / T); checked by a
  chi-square test, together with the two temperature limits.
* The page's clamp: draws below 1e-10 count as 1e-10.
* Softmax is shift invariant: adding a constant to a row's logits does not
  change the sample.
"""
import math

import numpy as np
import pytest

from oracle import sampler as S


def _bf16(x):
    u = np.asarray(x, dtype=np.float32).view(np.uint32)
    return ((u + ((u >> 16) & 1) + 0x7FFF) >> 16).astype(np.uint16)


def test_unit_draws_give_the_greedy_argmax(S=S):
    rng = np.random.default_rng(1)
    logits = rng.standard_normal((9, 300)).astype(np.float32)
    logits[3, 17] = logits[3, 200] = 9.0  # a tie: the first maximum wins
    t = rng.uniform(0.3, 2.0, 9).astype(np.float32)
    tok, _ = S.sample_gumbel(logits, t, np.ones_like(logits))
    assert tok.tolist() == logits.argmax(axis=1).tolist()
    assert tok[3] == 17


def test_equal_logits_pick_the_smallest_draw(S=S):
    rng = np.random.default_rng(2)
    e = rng.standard_exponential((6, 50)).astype(np.float32)
    tok, _ = S.sample_gumbel(np.full((6, 50), 0.25, np.float32), np.ones(6, np.float32), e)
    assert tok.tolist() == e.argmin(axis=1).tolist()


def _chi2_sf(x, k):
    # survival function of chi-square with k degrees of freedom (k even), closed form
    assert k % 2 == 0
    term, s = 1.0, 1.0
    for i in range(1, k // 2):
        term *= (x / 2) / i
        s += term
    return math.exp(-x / 2) * s


@pytest.mark.parametrize("temp", [0.7, 1.3])
def test_sample_frequencies_follow_the_softmax(temp, S=S):
    logits = np.array([1.0, 0.2, -0.5, 2.0, 0.0, -1.5, 0.7], np.float32)
    n = 40000
    rng = np.random.default_rng(7)
    e = rng.standard_exponential((n, logits.size)).astype(np.float32)
    tok, _ = S.sample_gumbel(np.tile(logits, (n, 1)), np.full(n, temp, np.float32), e)
    counts = np.bincount(tok, minlength=logits.size)
    w = np.exp(logits.astype(np.float64) / temp)
    expect = n * w / w.sum()
    chi2 = float(((counts - expect) ** 2 / expect).sum())
    assert _chi2_sf(chi2, logits.size - 1) > 1e-4, (counts, expect)


def test_temperature_limits(S=S):
    logits = np.array([0.5, 2.0, -1.0, 1.0], np.float32)
    n = 20000
    rng = np.random.default_rng(8)
    e = rng.standard_exponential((n, 4)).astype(np.float32)
    hot, _ = S.sample_gumbel(np.tile(logits, (n, 1)), np.full(n, 1e4, np.float32), e)
    assert np.all(np.abs(np.bincount(hot, minlength=4) / n - 0.25) < 0.02)  # near uniform
    cold, _ = S.sample_gumbel(np.tile(logits, (n, 1)), np.full(n, 1e-3, np.float32), e)
    assert np.all(cold == 1)  # near greedy


def test_draws_are_clamped_at_1e_10(S=S):
    logits = np.log(np.array([[0.1, 0.3, 0.6]], np.float32))
    # Draws 0 and 1e-12 both count as 1e-10, so the larger probability wins.
    e = np.array([[1.0, 0.0, 1e-12]], np.float32)
    tok, _ = S.sample_gumbel(logits, np.ones(1, np.float32), e)
    assert tok[0] == 2
    e = np.array([[1.0, 1e-12, 0.0]], np.float32)
    tok, _ = S.sample_gumbel(logits, np.ones(1, np.float32), e)
    assert tok[0] == 2


def test_shift_invariance_and_bf16_input(S=S):
    rng = np.random.default_rng(9)
    x = rng.standard_normal((5, 1000)).astype(np.float32)
    e = rng.standard_exponential((5, 1000)).astype(np.float32)
    t = np.full(5, 0.8, np.float32)
    bits = _bf16(x)
    widened = (bits.astype(np.uint32) << 16).view(np.float32)
    a, _ = S.sample_gumbel(bits, t, e)
    b, _ = S.sample_gumbel(widened, t, e)
    c, _ = S.sample_gumbel(widened + np.float32(4.0), t, e)  # exact shift in fp32 for these magnitudes
    assert a.tolist() == b.tolist() == c.tolist()


def test_bad_temperature_is_refused(S=S):
    with pytest.raises(ValueError):
        S.sample_gumbel(np.zeros((1, 4), np.float32), np.zeros(1, np.float32), np.ones((1, 4), np.float32))


# Plausible mistakes planted in copies of the oracle: each must fail a pin.
MUTANTS = {
    "temperature dropped": ("x = x / t[:, None]", "x = x"),
    "temperature multiplied": ("x = x / t[:, None]", "x = x * t[:, None]"),
    "draws multiplied": ("q = p / np.maximum(", "q = p * np.maximum("),
    "divided by the constant e": ("q = p / np.maximum(np.asarray(exp_noise, dtype=np.float32), E_MIN)",
                                  "q = p / np.float32(np.e) + 0 * np.asarray(exp_noise, dtype=np.float32)"),
    "clamp dropped": ("np.maximum(np.asarray(exp_noise, dtype=np.float32), E_MIN)",
                      "np.asarray(exp_noise, dtype=np.float32)"),
    "argmin": ("return q.argmax(axis=1)", "return q.argmin(axis=1)"),
    "last maximum": ("return q.argmax(axis=1)", "return (q.shape[1] - 1 - q[:, ::-1].argmax(axis=1))"),
}
PINS = [test_unit_draws_give_the_greedy_argmax, test_equal_logits_pick_the_smallest_draw,
        lambda S: test_sample_frequencies_follow_the_softmax(0.7, S), test_temperature_limits,
        test_draws_are_clamped_at_1e_10, test_shift_invariance_and_bf16_input]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_every_mutant_fails_a_pin(name):
    import types
    src = open(S.__file__, encoding="utf-8").read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, name
    mod = types.ModuleType("sampler_mutant")
    exec(compile(src.replace(old, new), "sampler_mutant.py", "exec"), mod.__dict__)
    failed = 0
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin(S=mod)
        except (AssertionError, ValueError, FloatingPointError):
            failed += 1
    assert failed > 0, f"mutant '{name}' passes every pin"
