"""Gumbel-max sampling oracle (test infrastructure: only the tests, the smoke
check and the benchmark's CPU-baseline leg use it; the product library never
loads it).

[NV12 §12.2 "采样器"] Sampler.forward: the logits are widened to fp32 and
divided by the row's temperature, turned into probabilities by a softmax,
divided elementwise by Exp(1) draws clamped below at 1e-10, and the row's
first argmax is the sampled token.  The page computes in fp32, so this does
too (numpy float32), in the page's order: divide, softmax (subtract the row
max, exponentiate, normalise), divide, argmax.  The draws are an input: the
caller owns the random state, as the page's exponential_() call does.
"""
from __future__ import annotations

import numpy as np

E_MIN = np.float32(1e-10)


def _as_f32(logits) -> np.ndarray:
    a = np.asarray(logits)
    if a.dtype == np.uint16:  # bf16 bit patterns: the high half of an fp32
        return (a.astype(np.uint32) << 16).view(np.float32)
    return a.astype(np.float32)


def sample_gumbel(logits, temperatures, exp_noise):
    """Returns (tokens int32 [batch], q float32 [batch, vocab]) with
    q = softmax(logits / T) / max(E, 1e-10) and tokens = first argmax of q."""
    x = _as_f32(logits)
    t = np.asarray(temperatures, dtype=np.float32)
    if np.any(~(t > np.float32(1e-10))):
        raise ValueError("temperature must be > 1e-10 (the page asserts it)")
    x = x / t[:, None]
    m = x.max(axis=1, keepdims=True)
    e = np.exp(x - m)
    p = e / e.sum(axis=1, keepdims=True, dtype=np.float32)
    q = p / np.maximum(np.asarray(exp_noise, dtype=np.float32), E_MIN)
    return q.argmax(axis=1).astype(np.int32), q


def scores_f64(logits, temperatures, exp_noise) -> np.ndarray:
    """The same q in float64, for judging near-ties between two indices."""
    x = _as_f32(logits).astype(np.float64) / np.asarray(temperatures, dtype=np.float64)[:, None]
    x = x - x.max(axis=1, keepdims=True)
    p = np.exp(x)
    p /= p.sum(axis=1, keepdims=True)
    return p / np.maximum(np.asarray(exp_noise, dtype=np.float64), 1e-10)
