"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks an oracle function against something other than itself:
golden values (tests/golden, each with its citation), closed forms, a library
routine in a special case, brute force on tiny inputs, or an invariant the
pages state. The mutation tests plant a mistake in the oracle (on the CPU) and
check that at least one pin catches it.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from conftest import read_golden


# ---------------------------------------------------------------- numerics of storage types

def test_half_decode_matches_ieee_for_every_pattern():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits])
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.all(np.isnan(got[np.isnan(ref)]))
    assert np.array_equal(got[np.isinf(ref)], ref[np.isinf(ref)])


def test_bf16_rounding_matches_torch_round_to_nearest_even():
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-6, 6, 20000),
                        [0.0, -0.0, 1.0, -1.0, 3.0e38, 1e-40]]).astype(np.float32)
    # exact ties: mantissa pattern ...1000 0000 0000 0000 below the bf16 lsb
    u = rng.integers(0, 1 << 15, 2000).astype(np.uint32) << 16 | 0x8000
    u = (u | 0x3F800000) & 0x3FFFFFFF
    x = np.concatenate([x, u.view(np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_from_double(float(v)) for v in x], dtype=np.uint16)
    assert np.array_equal(got, ref)
    back = np.array([oracle.bf16_to_double(int(b)) for b in ref])
    assert np.array_equal(back, torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).float().numpy())


def test_bf16_rounding_goes_through_fp32():
    # 1 + 2^-8 + 2^-30: nearest bf16 from fp64 is 1 + 2^-7, but fp32 first rounds
    # the 2^-30 away, leaving an exact tie that rounds to even (1.0).
    x = 1.0 + 2.0 ** -8 + 2.0 ** -30
    assert oracle.bf16_to_double(oracle.bf16_from_double(x)) == 1.0


# ---------------------------------------------------------------- dequantisation

def _q4_from_groups(scale_bits, min_bits, codes_2d):
    rows, cols = codes_2d.shape
    packed = (codes_2d[:, 0::2] | (codes_2d[:, 1::2] << 4)).astype(np.uint8)
    return dict(codes=packed, scales=np.asarray(scale_bits, np.uint16).reshape(rows, cols // 64).view(np.float16),
                mins=np.asarray(min_bits, np.uint16).reshape(rows, cols // 64).view(np.float16),
                rows=rows, cols=cols)


def test_dequant_hand_built_groups_golden():
    for sb, mb, code, exp in read_golden("dequant_groups.txt"):
        codes = np.full((1, 64), int(code), dtype=np.uint8)
        codes[0, 1::2] = (int(code) + 1) % 16       # odd elements: next code, high nibble
        t = _q4_from_groups([int(sb, 16)], [int(mb, 16)], codes)
        w = oracle.dequant_row(t, 0)
        assert w[0] == float(exp)
        s = oracle.half_to_double(int(sb, 16))
        m = oracle.half_to_double(int(mb, 16))
        assert w[1] == s * ((int(code) + 1) % 16) + m


def test_dequant_extremes_and_no_half_code():
    # codes 0 and 15 give min and 15*scale + min; with min = -7.5*scale the
    # dequantised values are symmetric and never zero (q = 7.5 is not a code)
    rng = np.random.default_rng(1)
    cfg = synth.workload(0)
    t = synth.make_weights(cfg)["L0.wq"]
    for r in rng.integers(0, t["rows"], 8):
        w = oracle.dequant_row(t, int(r))
        s = t["scales"][r].astype(np.float64).repeat(64)
        m = t["mins"][r].astype(np.float64).repeat(64)
        q = np.rint((w - m) / s)
        assert np.all((q >= 0) & (q <= 15))
        assert np.allclose(q * s + m, w, rtol=0, atol=0)
        assert np.all(np.abs(w) > 0)


def _dense(t):
    lo = t["codes"] & 15
    hi = t["codes"] >> 4
    q = np.empty((t["rows"], t["cols"]), dtype=np.float64)
    q[:, 0::2] = lo
    q[:, 1::2] = hi
    s = t["scales"].astype(np.float64).repeat(64, axis=1)
    m = t["mins"].astype(np.float64).repeat(64, axis=1)
    return s * q + m


@pytest.mark.parametrize("rows,cols", [(3, 64), (5, 128), (7, 5632), (33, 256)])
def test_matvec_equals_dense_brute_force(rows, cols):
    rng = np.random.default_rng(rows * 1000 + cols)
    t = synth._q4(rng, rows, cols)
    x = rng.standard_normal(cols)
    ref = _dense(t) @ x
    got = oracle.matvec(t, x)
    assert np.allclose(got, ref, rtol=1e-13, atol=1e-15 * np.abs(ref).max())


@pytest.mark.parametrize("mut", ["nibble_order", "scale_min_swap"])
def test_matvec_pin_catches_planted_mistakes(mut):
    rng = np.random.default_rng(3)
    t = synth._q4(rng, 5, 128)
    x = rng.standard_normal(128)
    ref = _dense(t) @ x
    with oracle.mutation(mut):
        got = oracle.matvec(t, x)
    assert not np.allclose(got, ref, rtol=1e-6)


# ---------------------------------------------------------------- RMSNorm, SiLU, argmax

def test_rmsnorm_closed_forms():
    n, eps = 256, 1e-5
    w = np.linspace(0.5, 1.5, n).astype(np.float32)
    for c in (0.3, -2.0, 7.0):
        got = oracle.rmsnorm(np.full(n, c), w, eps)
        assert np.allclose(got, np.sign(c) * w.astype(np.float64) / math.sqrt(1.0 + eps / c ** 2), rtol=1e-14)
    # eps = 0: scale invariance and unit root-mean-square with unit weights
    x = np.random.default_rng(0).standard_normal(n)
    ones = np.ones(n, np.float32)
    a = oracle.rmsnorm(x, ones, 0.0)
    assert np.allclose(a, oracle.rmsnorm(37.0 * x, ones, 0.0), rtol=1e-14)
    assert abs(np.sqrt(np.mean(a ** 2)) - 1.0) < 1e-14


def test_silu_mul_closed_forms():
    from scipy.special import expit
    z = np.linspace(-30, 30, 601)
    u = np.linspace(2, -1, 601)
    got = oracle.silu_mul(z, u)
    assert np.allclose(got, z * expit(z) * u, rtol=1e-14, atol=1e-300)
    assert oracle.silu_mul([0.0], [5.0])[0] == 0.0


def test_argmax_lowest_index_on_ties_and_nan():
    assert oracle.argmax_f32([1.0, 3.0, 3.0, 2.0]) == 1
    assert oracle.argmax_f32([-1.0, -1.0]) == 0
    # values equal after rounding to fp32 tie too
    assert oracle.argmax_f32([1.0, 1.0 + 1e-12, 0.5]) == 0
    assert oracle.argmax_f32([0.0, float("nan")]) == -1


# ---------------------------------------------------------------- RoPE

@pytest.mark.parametrize("neox", [0, 1])
def test_rope_identity_norms_and_composition(neox):
    hd, theta = 64, 1e4
    v = np.random.default_rng(2).standard_normal(hd)
    assert np.array_equal(oracle.rope(v, 0, theta, neox), v)
    pairs = [(i, i + hd // 2) if neox else (2 * i, 2 * i + 1) for i in range(hd // 2)]
    r = oracle.rope(v, 37, theta, neox)
    for a, b in pairs:
        assert abs(math.hypot(r[a], r[b]) - math.hypot(v[a], v[b])) < 1e-12
    # first pair rotates by exactly pos radians (theta_0 = 1)
    a, b = pairs[0]
    assert abs(r[a] - (v[a] * math.cos(37) - v[b] * math.sin(37))) < 1e-12
    # rotation by p equals p successive rotations by the position-1 angle
    s = v.copy()
    for _ in range(5):
        s = oracle.rope(s, 1, theta, neox)
    assert np.allclose(s, oracle.rope(v, 5, theta, neox), atol=1e-12)


def test_rope_pairing_layouts_differ():
    hd = 64
    e0 = np.zeros(hd)
    e0[0] = 1.0
    inter = oracle.rope(e0, 1, 1e4, 0)
    neox = oracle.rope(e0, 1, 1e4, 1)
    assert set(np.nonzero(np.abs(inter) > 1e-15)[0]) == {0, 1}
    assert set(np.nonzero(np.abs(neox) > 1e-15)[0]) == {0, hd // 2}


@pytest.mark.parametrize("mut", ["rope_pairing", "rope_sign"])
def test_rope_pins_catch_planted_mistakes(mut):
    hd = 64
    e0 = np.zeros(hd)
    e0[0] = 1.0
    with oracle.mutation(mut):
        got = oracle.rope(e0, 1, 1e4, 0)
    expected = np.zeros(hd)
    expected[0], expected[1] = math.cos(1.0), math.sin(1.0)
    assert not np.allclose(got, expected, atol=1e-12)


# ---------------------------------------------------------------- attention

def _bf16(a):
    return synth.bf16_bits_from_f32(np.asarray(a, np.float32))


def test_attention_single_entry_returns_v_exactly():
    rng = np.random.default_rng(4)
    for hd in (64, 128):
        k = _bf16(rng.standard_normal((1, hd)))
        v = _bf16(rng.standard_normal((1, hd)))
        out = oracle.attend(rng.standard_normal(hd), k, v)
        vv = np.array([oracle.bf16_to_double(int(b)) for b in v[0]])
        assert np.array_equal(out, vv)


def test_attention_uniform_keys_give_mean_of_values():
    rng = np.random.default_rng(5)
    hd, n = 64, 19
    k = np.repeat(_bf16(rng.standard_normal((1, hd))), n, axis=0)
    v = _bf16(rng.standard_normal((n, hd)))
    out = oracle.attend(rng.standard_normal(hd), k, v)
    vv = np.array([[oracle.bf16_to_double(int(b)) for b in row] for row in v])
    assert np.allclose(out, vv.mean(axis=0), rtol=1e-13, atol=1e-15)


def test_attention_two_positions_closed_form():
    hd = 64
    q = np.zeros(hd)
    q[0] = 8.0                                # score_t = 8 * k_t[0] / 8 = k_t[0]
    k = _bf16(np.array([[1.0] + [0.0] * 63, [3.0] + [0.0] * 63]))
    v = _bf16(np.array([[2.0] * hd, [-4.0] * hd]))
    out = oracle.attend(q, k, v)
    p1 = 1.0 / (1.0 + math.exp(2.0))          # softmax(1, 3)
    assert np.allclose(out, p1 * 2.0 + (1 - p1) * -4.0, rtol=1e-14)


# ---------------------------------------------------------------- whole decoder

def _tiny_cfg(**kw):
    cfg = dict(index=90, name="brute", dim=128, n_layers=2, n_heads=4, n_kv_heads=2, head_dim=32,
               ffn_dim=192, vocab=64, norm_eps=1e-5, rope_theta=1e4, rope_neox=0, qk_norm=0,
               tied=0, prompt_len=5, decode_steps=3, batch=1, prefill_kv=0)
    cfg.update(kw)
    return cfg


def _bf16_of(x):
    """bf16 storage of fp64 values, rounded through fp32 as the pages append from f32."""
    return torch.from_numpy(np.asarray(x, np.float64)).float().to(torch.bfloat16).double().numpy()


def _brute_forward(cfg, w, toks):
    """Dense numpy restatement of the decoder (prefill of all positions, causal)."""
    d, hd, Hq, Hkv = cfg["dim"], cfg["head_dim"], cfg["n_heads"], cfg["n_kv_heads"]
    n, eps = len(toks), cfg["norm_eps"]
    emb = w["embed"]
    if emb["kind"] == "bf16":
        E = torch.from_numpy(emb["data"].view(np.int16)).view(torch.bfloat16).double().numpy()
    else:
        E = emb["data"].astype(np.float64)

    def norm(x, g):
        return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * g.astype(np.float64)

    def rot(x, pos):                          # x [n, heads, hd]
        i = np.arange(hd // 2)
        ang = pos[:, None] * cfg["rope_theta"] ** (-2.0 * i / hd)
        c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
        if cfg["rope_neox"]:
            a, b = x[..., : hd // 2], x[..., hd // 2:]
            return np.concatenate([a * c - b * s, a * s + b * c], axis=-1)
        a, b = x[..., 0::2], x[..., 1::2]
        out = np.empty_like(x)
        out[..., 0::2] = a * c - b * s
        out[..., 1::2] = a * s + b * c
        return out

    h = E[np.asarray(toks)]
    pos = np.arange(n, dtype=np.float64)
    for l in range(cfg["n_layers"]):
        W = {k: _dense(w[f"L{l}.{k}"]) for k in ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")}
        xn = norm(h, w[f"L{l}.attn_norm"]["data"])
        q = (xn @ W["wq"].T).reshape(n, Hq, hd)
        k = (xn @ W["wk"].T).reshape(n, Hkv, hd)
        v = (xn @ W["wv"].T).reshape(n, Hkv, hd)
        if cfg["qk_norm"]:
            q = norm(q, w[f"L{l}.q_norm"]["data"])
            k = norm(k, w[f"L{l}.k_norm"]["data"])
        q, k = rot(q, pos), rot(k, pos)
        k, v = _bf16_of(k), _bf16_of(v)
        rep = Hq // Hkv
        k = np.repeat(k, rep, axis=1)         # _repeat_kv: head h uses kv head h // rep
        v = np.repeat(v, rep, axis=1)
        s = np.einsum("thd,jhd->htj", q, k) / math.sqrt(hd)
        s = np.where(np.tril(np.ones((n, n), bool))[None], s, -np.inf)
        p = np.exp(s - s.max(-1, keepdims=True))
        p /= p.sum(-1, keepdims=True)
        o = np.einsum("htj,jhd->thd", p, v).reshape(n, Hq * hd)
        h = h + o @ W["wo"].T
        xn = norm(h, w[f"L{l}.ffn_norm"]["data"])
        g, u = xn @ W["w_gate"].T, xn @ W["w_up"].T
        h = h + (g / (1 + np.exp(-g)) * u) @ W["w_down"].T
    xn = norm(h, w["final_norm"]["data"])
    lm = E if cfg["tied"] else _dense(w["lm_head"])
    return xn @ lm.T


@pytest.mark.parametrize("variant", [dict(), dict(rope_neox=1, qk_norm=1, tied=1, rope_theta=1e6),
                                     dict(n_heads=8, n_kv_heads=2, head_dim=16)])
def test_decoder_matches_dense_brute_force(variant):
    cfg = _tiny_cfg(**variant)
    w = synth.make_weights(cfg, seed=123)
    toks = synth.make_prompt(cfg, seed=9, n=7)
    ref = _brute_forward(cfg, w, toks)
    m = oracle.OracleModel(cfg, w)
    cache = m.new_cache(16)
    got = np.array([m.step(cache, int(t)) for t in toks])
    assert np.allclose(got, ref, rtol=1e-9, atol=1e-11 * np.abs(ref).max())
    assert np.allclose(m.full_prefix(toks), ref, rtol=1e-9, atol=1e-11 * np.abs(ref).max())


@pytest.mark.parametrize("mut", ["gqa_map", "no_residual", "rope_pairing", "qk_orientation",
                                 "mask_polarity", "cache_frontier"])
def test_decoder_pins_catch_planted_mistakes(mut):
    cfg = _tiny_cfg(n_heads=8, n_kv_heads=2, head_dim=16)
    w = synth.make_weights(cfg, seed=123)
    toks = synth.make_prompt(cfg, seed=9, n=7)
    ref = _brute_forward(cfg, w, toks)
    m = oracle.OracleModel(cfg, w)
    with oracle.mutation(mut):
        cache = m.new_cache(16)
        cached = np.array([m.step(cache, int(t)) for t in toks])
        full = m.full_prefix(toks)
    tol = dict(rtol=1e-9, atol=1e-11 * np.abs(ref).max())
    caught = (not np.allclose(cached, ref, **tol)) or (not np.allclose(full, ref, **tol)) \
        or (not np.array_equal(cached, full))
    assert caught


def test_prefix_equals_cache_bit_identical_every_position():
    # pytensor-ml issue, acceptance rules: cached output matches full-prefix
    # output on all logits at every tested step
    cfg = synth.workload(0)
    w = synth.make_weights(cfg)
    m = oracle.OracleModel(cfg, w)
    toks = synth.make_prompt(cfg)
    cache = m.new_cache(32)
    cached = np.array([m.step(cache, int(t)) for t in toks])
    full = m.full_prefix(toks)
    assert np.array_equal(cached, full)


def test_one_token_append_writes_one_slot():
    # pytensor-ml issue: a one-token append does not write over the whole cache
    cfg = synth.workload(0)
    m = oracle.OracleModel(cfg, synth.make_weights(cfg))
    cache = m.new_cache(40)
    cache.k[...] = 0xABCD
    cache.v[...] = 0xABCD
    for t in synth.make_prompt(cfg)[:5]:
        m.step(cache, int(t))
    touched = np.any(cache.k != 0xABCD, axis=(0, 1, 3))
    assert list(np.nonzero(touched)[0]) == [0, 1, 2, 3, 4]


def test_shapes_match_printed_sizes():
    g = {k: float(v) for k, v in read_golden("model_shapes.txt")}
    c1 = synth.workload(1)
    assert (c1["dim"], c1["ffn_dim"], c1["n_layers"], c1["n_heads"], c1["n_kv_heads"], c1["vocab"]) == \
        tuple(int(g["tinyllama." + k]) for k in ("dim", "ffn", "layers", "heads", "kv_heads", "vocab"))
    def n_params(cfg):
        n = sum(o * i for _, o, i in synth.linear_shapes(cfg)) + cfg["vocab"] * cfg["dim"]
        n += cfg["n_layers"] * 2 * cfg["dim"] + cfg["dim"]
        if cfg["qk_norm"]:
            n += cfg["n_layers"] * 2 * cfg["head_dim"]
        return n
    assert abs(n_params(c1) / 1e9 - g["tinyllama.params_billion"]) < 0.0005
    c2 = synth.workload(2)
    assert abs(n_params(c2) * 4 / g["qwen3_0.6b.bytes_per_token_f32"] - 1) < 0.005
    assert abs(n_params(c2) * 2 / g["qwen3_0.6b.bytes_per_token_bf16"] - 1) < 0.005
