"""Pins of the oracle's 4-bit x int8 matvec (oracle/w4a8.py, the W4A8 row) on the CPU.

Against the pinned fp64 matvec where the quantization is exact (inputs on the
int8 grid of power-of-two block scales), against a hand-computed block, and
within the scheme's error class on random inputs.
"""
import numpy as np

import oracle
from oracle import w4a8
import synth


def _weights(rows, cols, seed):
    rng = np.random.default_rng(seed)
    return synth._q4(rng, rows, cols)


def test_exact_where_the_activations_sit_on_the_int8_grid():
    t = _weights(37, 256, 1)
    rng = np.random.default_rng(2)
    c = rng.integers(-127, 128, 256)
    e = rng.integers(-8, 3, 256 // 32)
    c[::32] = 127  # each block's largest magnitude sets its scale to 2^e exactly
    x = c * np.repeat(2.0 ** e, 32)
    y = w4a8.matvec(t, x)
    ref = oracle.matvec(t, x)
    assert np.allclose(y, ref, rtol=1e-13, atol=1e-13 * np.abs(ref).max())


def test_one_hand_computed_block():
    t = dict(kind="q4", rows=1, cols=64, codes=np.full((1, 32), 0x21, np.uint8),  # codes 1, 2, 1, 2, ...
             scales=np.array([[0.5]], np.float16), mins=np.array([[-1.0]], np.float16))
    x = np.zeros(64)
    x[0:32] = 127.0 * 0.25  # block 0: scale 0.25, codes 127
    x[32] = 127.0            # block 1: scale 1, code 127 at its first element, zeros after
    # block 0: S1 = 16*1*127 + 16*2*127, S2 = 32*127 -> 0.25*(0.5*S1 - S2); block 1: S1 = 127, S2 = 127
    expect = 0.25 * (0.5 * (48 * 127) - 32 * 127) + 1.0 * (0.5 * 127 - 127)
    assert w4a8.matvec(t, x)[0] == expect
    assert oracle.matvec(t, x)[0] == expect  # and the exact product agrees on this grid input


def test_random_inputs_stay_in_the_scheme_error_class():
    t = _weights(512, 2048, 3)
    rng = np.random.default_rng(4)
    x = rng.standard_normal(2048)
    y = w4a8.matvec(t, x)
    ref = oracle.matvec(t, x)
    rel = np.linalg.norm(y - ref) / np.linalg.norm(ref)
    assert 1e-5 < rel < 2e-2  # quantized, but only by the int8 blocks of x
