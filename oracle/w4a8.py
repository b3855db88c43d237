"""4-bit weights x int8 activations -- TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

The CPU scheme of the aot-llm page (implementation notes: "Per matmul, the
f32 activation vector is quantized once to Q8_0 ... and every output row is
an integer dot product scaled back to f32, the same scheme ggml uses"),
restated for this build's group-64 affine weights (w = scale * q + min,
q in 0..15):

* x is quantized once with the grouped int8 quantizer of the oracle
  (blocks of 32, fp16 scale d_b = fp16(amax / 127), codes c_j);
* each 64-input weight group covers two activation blocks; per block b the
  integer sums S1 = sum q_j c_j and S2 = sum c_j are exact, and the row
  gathers d_b * (scale * S1 + min * S2) in fp64.
"""
from __future__ import annotations

import numpy as np

from . import Q8_GROUP, q8_quantize

GROUP = 64


def unpack_codes(t: dict) -> np.ndarray:
    """Canonical 4-bit codes [rows][cols]: element 2j in the low nibble of byte j."""
    b = np.asarray(t["codes"], dtype=np.uint8)
    out = np.empty((b.shape[0], b.shape[1] * 2), dtype=np.int64)
    out[:, 0::2] = b & 0x0F
    out[:, 1::2] = b >> 4
    return out


def matvec(t: dict, x) -> np.ndarray:
    """y = W x with x quantized to grouped int8 and integer block dots."""
    rows, cols = int(t["rows"]), int(t["cols"])
    x = np.ascontiguousarray(x, dtype=np.float64)
    assert x.shape == (cols,) and cols % GROUP == 0
    c, d_bits = q8_quantize(x)
    d = np.asarray(d_bits, dtype=np.uint16).view(np.float16).astype(np.float64)  # exact
    q = unpack_codes(t)
    s = np.asarray(t["scales"]).astype(np.float64)
    m = np.asarray(t["mins"]).astype(np.float64)
    nb = cols // Q8_GROUP
    cb = c.astype(np.int64).reshape(nb, Q8_GROUP)
    qb = q.reshape(rows, nb, Q8_GROUP)
    S1 = np.einsum("rbj,bj->rb", qb, cb)   # integer, exact
    S2 = cb.sum(axis=1)                    # integer, exact
    g = np.arange(nb) // (GROUP // Q8_GROUP)
    terms = d[None, :] * (s[:, g] * S1 + m[:, g] * S2[None, :])
    y = np.zeros(rows)
    for b in range(nb):  # blocks in input order
        y += terms[:, b]
    return y
