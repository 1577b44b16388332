"""The sampler (temperature, softmax, Gumbel-max), restated on the CPU.

Test infrastructure only (see the package docstring).

[UML] §2.4 Model Runner: sampling is temperature, then softmax, then a
Gumbel-max draw; [LIFE] §4: the sampler runs on each sequence's last-position
logits and returns one token id per sequence.  The noise is passed in: E is a
(B, V) array of Exp(1) draws.

Readings where the pages are silent:
  * "Gumbel-max" is the exponential race argmax_i p_i / E_i, E_i ~ Exp(1),
    which equals argmax_i (x_i - ln E_i) because softmax is monotone in x;
  * E is clamped below at 1e-10 before it is used;
  * ties go to the lowest index;
  * a temperature that is not a positive finite number is a precondition
    violation: the row returns token 0 and is reported.

In-kernel noise (the library's second sampler entry point) uses the
counter-based generator Philox4x32-10 of Salmon, Moraes, Dror and Shaw,
"Parallel random numbers: as easy as 1, 2, 3" (SC 2011), restated below from
that definition.  `philox4x32_10` is pinned to the published known-answer
vectors of that generator (the known-answer file of the authors' Random123
library, stored under tests/golden/); the stream built on it is further checked
by inverting its round function, by statistics of its output, and through the
Gumbel-max law of the draws it feeds.
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


# ----------------------------------------------------------------------------
# counter-based Exp(1) noise
# ----------------------------------------------------------------------------
PHILOX_M = (0xD2511F53, 0xCD9E8D57)       # round multipliers
PHILOX_W = (0x9E3779B9, 0xBB67AE85)       # key schedule increments (Weyl sequence)
MASK32 = 0xFFFFFFFF


def philox_round(c, k0, k1):
    """One Philox4x32 round on counters c (N, 4) of 32-bit values held in
    uint64: multiply words 0 and 2 by the two constants, split each 64-bit
    product into (hi, lo), and output (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0)."""
    p0 = np.uint64(PHILOX_M[0]) * c[:, 0]
    p1 = np.uint64(PHILOX_M[1]) * c[:, 2]
    hi0, lo0 = p0 >> np.uint64(32), p0 & np.uint64(MASK32)
    hi1, lo1 = p1 >> np.uint64(32), p1 & np.uint64(MASK32)
    return np.stack([hi1 ^ c[:, 1] ^ np.uint64(k0), lo1, hi0 ^ c[:, 3] ^ np.uint64(k1), lo0],
                    axis=1)


def philox4x32_10(counters, key):
    """Ten rounds; the 64-bit key (k0, k1) is bumped by the Weyl increments
    before every round after the first.  counters: (N, 4) integers < 2^32.
    Returns (N, 4) uint64 words < 2^32."""
    c = np.asarray(counters, dtype=np.uint64)
    k0, k1 = int(key[0]) & MASK32, int(key[1]) & MASK32
    for r in range(10):
        if r > 0:
            k0 = (k0 + PHILOX_W[0]) & MASK32
            k1 = (k1 + PHILOX_W[1]) & MASK32
        c = philox_round(c, k0, k1)
    return c


def philox_words(n, seed: int, offset: int):
    """Output word of entry n (a flat index): Philox4x32-10 keyed by the 64-bit
    seed on counter (n // 4 as two 32-bit words, offset as two 32-bit words),
    word n % 4."""
    n = np.asarray(n, dtype=np.uint64).reshape(-1)
    blk = n >> np.uint64(2)
    ctr = np.stack([blk & np.uint64(MASK32), blk >> np.uint64(32),
                    np.full_like(blk, offset & MASK32), np.full_like(blk, (offset >> 32) & MASK32)],
                   axis=1)
    w = philox4x32_10(ctr, (seed & MASK32, (seed >> 32) & MASK32))
    return w[np.arange(len(n)), (n & np.uint64(3)).astype(np.int64)]


def philox_exp_noise(batch: int, vocab: int, seed: int, offset: int):
    """(B, V) Exp(1) noise: entry n = row * vocab + i draws word w, U = (w >> 8
    plus one) * 2^-24 (exact, in (0, 1]) and E = -ln U (float64)."""
    n = np.arange(batch * vocab, dtype=np.uint64)
    w = philox_words(n, seed, offset)
    u = ((w >> np.uint64(8)) + np.uint64(1)).astype(np.float64) * 2.0 ** -24
    return (-np.log(u)).reshape(batch, vocab)


def sample_philox(logits, temperatures, seed: int, offset: int):
    """The draw of `sample` with the noise of `philox_exp_noise`."""
    lg = np.asarray(logits)
    E = philox_exp_noise(lg.shape[0], lg.shape[1], seed, offset)
    return sample(lg, temperatures, E)
