"""The sampler (temperature, softmax, Gumbel-max), restated on the CPU.

Test infrastructure only (see the package docstring).

[UML] §2.4 Model Runner: sampling is temperature, then softmax, then a
Gumbel-max draw; [LIFE] §4: the sampler runs on each sequence's last-position
logits and returns one token id per sequence.  The noise is passed in: E is a
(B, V) array of Exp(1) draws.

Readings where the pages are silent (listed in the design doc):
  * "Gumbel-max" is the exponential race argmax_i p_i / E_i, E_i ~ Exp(1),
    which equals argmax_i (x_i - ln E_i) because softmax is monotone in x;
  * E is clamped below at 1e-10 before it is used;
  * ties go to the lowest index;
  * a temperature that is not a positive finite number is a precondition
    violation: the row returns token 0 and is reported.
"""
from __future__ import annotations

import numpy as np

NOISE_FLOOR = 1e-10


def _row_ok(t: float) -> bool:
    return bool(np.isfinite(t) and t > 0.0)


def sample(logits, temperatures, exp_noise):
    """Step by step: x = logits / T; p = softmax(x) (max subtracted); key_i =
    p_i / E_i; token = first index of the largest key.  float64 throughout.
    Returns (token ids int32 (B,), list of rows with a bad temperature)."""
    lg = np.asarray(logits, dtype=np.float64)
    T = np.asarray(temperatures, dtype=np.float64).reshape(-1)
    E = np.asarray(exp_noise, dtype=np.float64)
    B = lg.shape[0]
    out = np.zeros(B, dtype=np.int32)
    bad = []
    for r in range(B):
        if not _row_ok(T[r]):
            bad.append(r)
            continue
        x = lg[r] / T[r]
        e = np.exp(x - x.max())
        p = e / e.sum()
        key = p / np.maximum(E[r], NOISE_FLOOR)
        out[r] = int(np.argmax(key))            # first maximum: lowest index
    return out, bad


def sample_key_form(logits, temperatures, exp_noise):
    """The same draw as `sample`, written as argmax_i (x_i - ln E_i).  The
    tests require both statements to agree.  Returns (ids, keys) where keys is
    the (B, V) float64 array of x_i - ln E_i (rows with a bad temperature are
    -inf)."""
    lg = np.asarray(logits, dtype=np.float64)
    T = np.asarray(temperatures, dtype=np.float64).reshape(-1)
    E = np.asarray(exp_noise, dtype=np.float64)
    keys = np.full(lg.shape, -np.inf)
    out = np.zeros(lg.shape[0], dtype=np.int32)
    for r in range(lg.shape[0]):
        if not _row_ok(T[r]):
            continue
        keys[r] = lg[r] / T[r] - np.log(np.maximum(E[r], NOISE_FLOOR))
        out[r] = int(np.argmax(keys[r]))
    return out, keys


def near_ties(keys: np.ndarray, rel: float = 1e-5):
    """Per row, the indices whose key lies within rel*max(1,|top|) of the row's
    top key.  A row with more than one such index is one where a float32
    evaluation may legitimately pick a different index than float64."""
    out = []
    for r in range(keys.shape[0]):
        row = keys[r]
        top = row.max()
        tol = rel * max(1.0, abs(top)) if np.isfinite(top) else 0.0
        out.append(np.flatnonzero(row >= top - tol))
    return out
