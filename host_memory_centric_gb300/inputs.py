"""Seeded synthetic inputs (token ids).  Holds none of the training arithmetic.

Token ids are uniform in [0, V), drawn from a counter-based SplitMix64 stream
(Steele, Lea and Flood 2014): the i-th output of the stream seeded with s is
mix(s + (i+1)*0x9E3779B97F4A7C15), with the variant-13 finaliser.  The step's
stream key is output number ``step`` of the token seed's stream, and id i is
``((out(key, i) >> 32) * V) >> 32`` (multiply-shift range reduction).  The
layout is [micro][batch][seq].  The pages trained on MetaMathQA; the speed
of a dense causal decoder does not depend on the token values, so these ids
stand in for it with the same shapes.
"""
from __future__ import annotations

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def splitmix64(seed: int, idx: np.ndarray) -> np.ndarray:
    """Outputs number ``idx`` (uint64 array) of the stream seeded with ``seed``."""
    with np.errstate(over="ignore"):
        z = np.uint64(seed) + (idx.astype(np.uint64) + np.uint64(1)) * _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def tokens(seed: int, step: int, micro: int, batch: int, seq: int, vocab: int) -> np.ndarray:
    key = int(splitmix64(seed, np.array([step], dtype=np.uint64))[0])
    n = micro * batch * seq
    r = splitmix64(key, np.arange(n, dtype=np.uint64))
    with np.errstate(over="ignore"):
        ids = ((r >> np.uint64(32)) * np.uint64(vocab)) >> np.uint64(32)
    return ids.astype(np.int32).reshape(micro, batch, seq)


def tokens_for(cfg: dict, step: int, seed: int = 1234) -> np.ndarray:
    return tokens(seed, step, cfg["micro"], cfg["batch"], cfg["seq"], cfg["vocab"])
