"""Pins of the oracle's grouped int8 K/V storage (the grouped-Q8 cache row).

fp16 scale conversion against numpy's IEEE half; the quantizer against closed
forms (grid values round-trip, halves round away from zero, the largest
magnitude maps to +-127, a zero group, the error bound, sign symmetry); the
int8 attention against the pinned bf16 attention where both stores hold the
same values; and the decoder's cached and full-prefix modes against each other.
"""
import numpy as np
import pytest

import oracle
import synth


def test_half_from_float_is_ieee_rne():
    rng = np.random.default_rng(11)
    xs = np.concatenate([rng.standard_normal(4000) * 10.0 ** rng.uniform(-9, 5, 4000),
                         [0.0, -0.0, 1.0, 65504.0, 65519.0, 65520.0, 6.1e-5, 5.96e-8, 2.98e-8, 1e-9, 1.0 + 2 ** -11,
                          1.0 + 3 * 2 ** -11]]).astype(np.float32)
    with np.errstate(over="ignore"):  # values beyond fp16's range become infinity on both sides
        for x in xs:
            assert oracle.half_from_float(float(x)) == int(np.float16(x).view(np.uint16)), x


def _scale(d_bits):
    return oracle.half_to_double(int(d_bits))


def test_grid_values_round_trip_and_amax_is_127():
    for d in (2.0 ** -6, 0.0078125 * 3, 1.5, 0.25):  # fp16-exact scales with 127*d exact in fp32
        j = np.arange(-127, 128)[::8]
        x = np.resize(j, 32).astype(np.float64) * d
        x[5] = 127 * d  # the group's largest magnitude
        q, dd = oracle.q8_quantize(x)
        assert _scale(dd[0]) == d
        assert np.array_equal(q.astype(np.float64) * d, x)
        assert q[5] == 127


def test_halves_round_away_from_zero_and_signs_mirror():
    d = 2.0 ** -4
    x = np.zeros(32)
    x[0] = 127 * d
    x[1:9] = (np.array([0, 1, 2, 3, 10, 50, 100, 125]) + 0.5) * d
    x[9:17] = -x[1:9]
    q, dd = oracle.q8_quantize(x)
    assert _scale(dd[0]) == d
    assert list(q[1:9]) == [1, 2, 3, 4, 11, 51, 101, 126]
    assert np.array_equal(q[9:17], -q[1:9])
    qn, _ = oracle.q8_quantize(-x)
    assert np.array_equal(qn, -q)


def test_zero_group_and_error_bound():
    q, dd = oracle.q8_quantize(np.zeros(64))
    assert not q.any() and not dd.any()
    rng = np.random.default_rng(12)
    for _ in range(50):
        x = rng.standard_normal(128) * 10.0 ** rng.uniform(-3, 2)
        q, dd = oracle.q8_quantize(x)
        xf = x.astype(np.float32).astype(np.float64)  # values are quantized from fp32
        for g in range(4):
            d = _scale(dd[g])
            amax = np.abs(xf[32 * g:32 * g + 32]).max()
            # fp16 rounding of amax/127: half an ulp (11 bits), or half the subnormal spacing 2^-24
            assert abs(d - amax / 127) <= max(amax / 127 * 2 ** -11, 2 ** -25) * (1 + 2 ** -20)
            err = np.abs(q[32 * g:32 * g + 32] * d - xf[32 * g:32 * g + 32])
            # half a step, plus what a scale rounded down leaves at the clamped end
            assert err.max() <= d / 2 + 127 * max(0.0, amax / 127 - d) + 1e-12 * amax


def test_int8_attention_equals_bf16_attention_on_shared_values():
    # codes times a power of two have at most 7 significant bits: exactly bf16
    rng = np.random.default_rng(13)
    n, hd = 9, 64
    k8 = rng.integers(-127, 128, (n, hd)).astype(np.int8)
    v8 = rng.integers(-127, 128, (n, hd)).astype(np.int8)
    ks = np.full((n, hd // 32), int(np.float16(2.0 ** -6).view(np.uint16)), np.uint16)
    vs = np.full((n, hd // 32), int(np.float16(2.0 ** -3).view(np.uint16)), np.uint16)
    to_bf16 = lambda a: (a.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    kb = to_bf16(k8.astype(np.float64) * 2.0 ** -6)
    vb = to_bf16(v8.astype(np.float64) * 2.0 ** -3)
    q = rng.standard_normal(hd)
    ref = oracle.attend(q, kb, vb)
    assert np.array_equal(oracle.attend_q8(q, k8, ks, v8, vs), ref)
    # one position: the stored value row itself
    one = oracle.attend_q8(q, k8[:1], ks[:1], v8[:1], vs[:1])
    assert np.array_equal(one, v8[0].astype(np.float64) * 2.0 ** -3)


def test_cached_equals_full_prefix_with_int8_kv():
    cfg = synth.workload(0)
    w = synth.make_weights(cfg)
    prompt = synth.make_prompt(cfg)[:9]
    om = oracle.OracleModel(cfg, w)
    cache = om.new_cache(len(prompt), kv="q8")
    cached = np.array([om.step(cache, int(t)) for t in prompt])
    with oracle.kv_q8():
        full = om.full_prefix(prompt)
    assert np.array_equal(cached, full)
    # and the int8 store is a perturbation of the bf16 one, not another model
    bf = om.full_prefix(prompt)
    rel = np.abs(full - bf).max(axis=1) / np.abs(bf).max(axis=1)
    assert 0 < rel.max() < 0.05


def test_prefilled_int8_cache_holds_grid_rows_exactly():
    # pre-filled rows whose values are codes times a power of two, with a
    # largest code of 127 in every group: the int8 cache must hold exactly
    # those codes at (layer, head, position), with the power of two as scale
    cfg = synth.workload(0)
    rng = np.random.default_rng(21)
    n, H, hd, L = 12, cfg["n_kv_heads"], cfg["head_dim"], cfg["n_layers"]
    c8 = oracle.OracleCache(cfg, n + 3, kv="q8")
    to_bf16 = lambda a: (a.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    for l in range(L):
        codes = [rng.integers(-127, 128, (n, H, hd)) for _ in range(2)]
        for c in codes:
            c[:, :, ::32] = np.where(rng.random((n, H, hd // 32)) < 0.5, 127, -127)
        e = (-5 - l, -2 + l)
        c8.fill(l, to_bf16(codes[0] * 2.0 ** e[0]), to_bf16(codes[1] * 2.0 ** e[1]), pos0=2)
        for c, stored, scales, ex in ((codes[0], c8.k8, c8.ks, e[0]), (codes[1], c8.v8, c8.vs, e[1])):
            assert np.array_equal(stored[l, :, 2:2 + n, :], np.transpose(c, (1, 0, 2)).astype(np.int8))
            assert np.all(scales[l, :, 2:2 + n, :] == int(np.float16(2.0 ** ex).view(np.uint16)))
            assert not stored[l, :, :2].any() and not stored[l, :, 2 + n:].any()
