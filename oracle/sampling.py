"""Sampled next-token choice -- TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

Plain Python/numpy restatement, fp64 unless noted, of the sampling options the
pages list for the generated runtime (aot-llm page, "Generated binary options":
temperature with 0 = greedy, top-k, top-p nucleus threshold, RNG seed) and of
the counter-based generator that supplies the draw:

* Philox4x32-10 as published by Salmon, Moraes, Dror and Shaw, "Parallel
  random numbers: as easy as 1, 2, 3" (SC 2011): 10 rounds of two 32x32->64
  multiplications by 0xD2511F53 and 0xCD9E8D57 with the Weyl key schedule
  0x9E3779B9, 0xBB67AE85. Pinned by the paper's known-answer vectors.
* The draw for the token after position `pos` of sequence `seq`: counter
  (pos, seq, 0, 0), key (seed mod 2^32, seed div 2^32); u = (x0 >> 8) / 2^24.
* Choice (the plainest reading of the options): keep the top_k largest logits
  (ties: lower token id first), p_j = softmax((l_j - l_max) / T) in that
  order, keep the shortest prefix whose cumulative probability reaches top_p,
  and return the first token of the prefix whose cumulative probability
  exceeds u times the prefix's total.
"""
from __future__ import annotations

import numpy as np

_M0, _M1 = 0xD2511F53, 0xCD9E8D57
_W0, _W1 = 0x9E3779B9, 0xBB67AE85
_MASK = 0xFFFFFFFF


def philox4x32_10(counter, key):
    """Philox4x32 with 10 rounds: four 32-bit words of output for a 128-bit counter and a 64-bit key."""
    c0, c1, c2, c3 = (int(x) & _MASK for x in counter)
    k0, k1 = (int(x) & _MASK for x in key)
    for r in range(10):
        if r:
            k0 = (k0 + _W0) & _MASK
            k1 = (k1 + _W1) & _MASK
        p0 = _M0 * c0
        p1 = _M1 * c2
        hi0, lo0 = p0 >> 32, p0 & _MASK
        hi1, lo1 = p1 >> 32, p1 & _MASK
        c0, c1, c2, c3 = (hi1 ^ c1 ^ k0) & _MASK, lo1, (hi0 ^ c3 ^ k1) & _MASK, lo0
    return c0, c1, c2, c3


def uniform(seed: int, seq: int, pos: int) -> float:
    """The draw in [0, 1) for the token that follows position `pos` of sequence `seq`."""
    x0 = philox4x32_10((pos, seq, 0, 0), (seed & _MASK, (seed >> 32) & _MASK))[0]
    return (x0 >> 8) / float(1 << 24)


def sample(logits, temperature: float, top_k: int, top_p: float, u: float):
    """Token chosen from fp32 logits; also returns the quantities that decide it.

    info: sorted candidate ids, their cumulative probabilities, the prefix
    length n and the target u * c[n-1] (a decision whose target or top_p lies
    within rounding of a cumulative boundary is ambiguous between precisions).
    """
    lg = np.asarray(logits, dtype=np.float32).astype(np.float64)
    assert temperature > 0 and 1 <= top_k <= lg.size and 0 < top_p <= 1
    order = sorted(range(lg.size), key=lambda i: (-lg[i], i))[:top_k]  # value desc, id asc
    v = lg[order]
    e = np.exp((v - v[0]) / temperature)
    p = e / e.sum()
    c = np.cumsum(p)
    n = int(np.argmax(c >= top_p)) + 1 if (c >= top_p).any() else top_k
    target = u * c[n - 1]
    j = next((i for i in range(n) if c[i] > target), n - 1)
    return order[j], {"ids": order, "cum": c, "n": n, "target": target}
