"""The grouped int8 K/V cache (LLM_KV_Q8) on the GPU against the oracle's int8 cache.

The oracle's cache (kv="q8") quantizes each appended (position, head) row of
k and v in groups of 32 (fp16 scale fp16(amax / 127), codes rounded half away
from zero and clamped to +-127, decided in fp32) and attends over the stored
code x scale values in fp64. The GPU does the same in fp32 from its own k and
v, so a code can differ by one where the two sides' values straddle a
rounding boundary; the bars are:
  * pre-filled rows (llm_kv_write from bf16): codes and scales bit-exact
    with the oracle's quantizer of the same bf16 values;
  * appended rows: every stored value within one quantum of the oracle's
    (the two roundings) plus the hidden-state class (2e-3 of the row's
    largest value: how far the GPU's fp32 k, v may lie from the oracle's
    before quantizing), and at least 99 % of the codes identical;
  * per-layer hidden states at rel. L2 2e-3, logits at 5e-3 x max|logit|
    (the fp32 bars), teacher-forced on the oracle's tokens.
"""
import numpy as np
import pytest
import torch

import bit_quantized_token_gb300 as bq
import oracle
import synth

pytestmark = pytest.mark.gpu

HIDDEN_RL2 = 2e-3
LOGIT_REL = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available()
    bq.build()
    oracle.build()


def rel_l2(a, b):
    return float(np.linalg.norm(np.asarray(a, np.float64) - b) / np.linalg.norm(b))


def _values(codes, scale_bits):
    s = np.asarray(scale_bits, np.uint16).view(np.float16).astype(np.float64)
    return codes.astype(np.float64) * np.repeat(s, 32, axis=-1)


def _teacher_forced(cfg, m, om, cache, toks, n_check_from=0):
    logits = np.empty(cfg["vocab"], np.float32)
    worst = 0.0
    for i, tok in enumerate(toks):
        ref, ref_h = om.step(cache, int(tok), hidden=True)
        m.decode_step(0, int(tok), logits)
        if i < n_check_from:
            continue
        err = np.abs(logits - ref).max() / np.abs(ref).max()
        worst = max(worst, err)
        assert err <= LOGIT_REL, f"step {i}: logit error {err:.3e}"
        hid = m.hidden()
        for l in range(cfg["n_layers"] + 1):
            r = rel_l2(hid[l], ref_h[l])
            assert r <= HIDDEN_RL2, f"step {i} layer {l}: hidden rel L2 {r:.3e}"
    return worst


def _appended_rows_match(cfg, m, cache, pos0, n, seq=0):
    H, hd = cfg["n_kv_heads"], cfg["head_dim"]
    same = total = 0
    for l in range(cfg["n_layers"]):
        k, ks, v, vs = m.kv_read_q8(seq, l, pos0, n)
        for got_c, got_s, ref_c, ref_s, name in ((k, ks, cache.k8, cache.ks, "K"), (v, vs, cache.v8, cache.vs, "V")):
            rc = np.transpose(ref_c[l, :, pos0:pos0 + n], (1, 0, 2))
            rs = np.transpose(ref_s[l, :, pos0:pos0 + n], (1, 0, 2))
            gv, rv = _values(got_c, got_s), _values(rc, rs)
            quantum = np.repeat(np.maximum(got_s.view(np.float16), rs.view(np.float16)).astype(np.float64), 32, -1)
            # one quantum from the two roundings, plus how far the GPU's fp32 k, v may lie from the
            # oracle's before quantizing (the hidden-state class, 2e-3, of the row's largest value)
            tol = quantum * (1 + 1e-6) + HIDDEN_RL2 * np.abs(rv).max(axis=-1, keepdims=True)
            bad = np.argwhere(np.abs(gv - rv) > tol)
            assert bad.size == 0, (f"layer {l} {name}: appended values off at {bad[:4].tolist()}: gpu "
                                   f"{[float(gv[tuple(b)]) for b in bad[:4]]}, oracle {[float(rv[tuple(b)]) for b in bad[:4]]}, "
                                   f"quantum {[float(quantum[tuple(b)]) for b in bad[:4]]}")
            same += int((got_c == rc).sum())
            total += got_c.size
    assert same >= 0.99 * total, f"only {same} of {total} appended codes equal the oracle's"


@pytest.mark.parametrize("cfg", [synth.workload(0), synth.workload(1, n_layers=2, vocab=4096),
                                 synth.workload(2, n_layers=2, vocab=4096)],
                         ids=["tiny", "tinyllama-shape-2-layers", "qwen3-shape-2-layers"])
def test_kv8_decode_matches_the_oracle_int8_cache(cfg):
    w = synth.make_weights(cfg)
    prompt = synth.make_prompt(cfg)
    n = 24
    om = oracle.OracleModel(cfg, w)
    toks = list(prompt) + list(synth.make_prompt(cfg, seed=5, n=n))
    cache = om.new_cache(len(toks) + 1, kv="q8")
    with bq.Model(cfg, w, max_seq=len(toks) + 1, flags=bq.LLM_KV_Q8) as m:
        st = m.stats()
        hd, H, L = cfg["head_dim"], cfg["n_kv_heads"], cfg["n_layers"]
        assert st["kv_bytes_per_pos"] == 2 * L * H * (hd + hd // 16)
        _teacher_forced(cfg, m, om, cache, toks)
        assert m.kv_len(0) == len(toks)
        _appended_rows_match(cfg, m, cache, 0, len(toks))


def test_kv8_prefilled_rows_are_the_oracle_quantizer_bit_exactly():
    cfg = synth.workload(2, n_layers=2, vocab=4096)
    w = synth.make_weights(cfg)
    n_pre = 300
    with bq.Model(cfg, w, max_seq=n_pre + 4, flags=bq.LLM_KV_Q8) as m:
        for l in range(cfg["n_layers"]):
            kb, vb = synth.make_prefilled_kv(cfg, l, 0, n_pre)
            m.kv_write(0, l, 0, kb, vb)
            k, ks, v, vs = m.kv_read_q8(0, l, 0, n_pre)
            for got_c, got_s, bits in ((k, ks, kb), (v, vs, vb)):
                vals = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
                c, d = oracle.q8_quantize(vals.reshape(-1))
                assert np.array_equal(got_c.reshape(-1), c)
                assert np.array_equal(got_s.reshape(-1), d)
        with pytest.raises(bq.LlmError) as e:
            m.kv_read(0, 0, 0, 4)
        assert e.value.code == -2


@pytest.mark.parametrize("n_steps", [64])
def test_kv8_long_context_teacher_forced(n_steps):
    # 4096 pre-filled positions (the long-context workload) through the int8 cache
    cfg = synth.workload(3)
    w = synth.make_weights(cfg)
    n_pre = cfg["prefill_kv"]
    cap = n_pre + n_steps + 1
    om = oracle.OracleModel(cfg, w)
    cache = om.new_cache(cap, kv="q8")
    with bq.Model(cfg, w, max_seq=cap, flags=bq.LLM_KV_Q8) as m:
        for l in range(cfg["n_layers"]):
            k, v = synth.make_prefilled_kv(cfg, l, 0, n_pre)
            cache.fill(l, k, v)
            m.kv_write(0, l, 0, k, v)
        cache.set_len(n_pre)
        tok = int(synth.make_first_tokens(cfg, 1)[0])
        logits = np.empty(cfg["vocab"], np.float32)
        for i in range(n_steps):
            ref, ref_h = om.step(cache, tok, hidden=True)
            m.decode_step(0, tok, logits)
            err = np.abs(logits - ref).max() / np.abs(ref).max()
            assert err <= LOGIT_REL, f"step {i}: logit error {err:.3e}"
            if i % 8 == 0:
                hid = m.hidden()
                for l in range(cfg["n_layers"] + 1):
                    assert rel_l2(hid[l], ref_h[l]) <= HIDDEN_RL2, f"step {i} layer {l}"
            tok = oracle.argmax_f32(ref)
        _appended_rows_match(cfg, m, cache, n_pre, n_steps)


@pytest.mark.parametrize("cfg,n_prompt", [(synth.workload(0), 70), (synth.workload(2, n_layers=2, vocab=4096), 45)],
                         ids=["tiny-3-chunks", "qwen3-shape-2-layers"])
def test_kv8_batched_prefill_matches_token_by_token(cfg, n_prompt):
    # batched prompt processing into the int8 cache against the oracle's
    # token-by-token prefill into its int8 cache: last logits and greedy
    # token, every appended row, then greedy decoding from that cache
    w = synth.make_weights(cfg)
    prompt = synth.make_prompt(cfg, n=n_prompt)
    n = 8
    cap = n_prompt + n + 1
    om = oracle.OracleModel(cfg, w)
    cache = om.new_cache(cap, kv="q8")
    ref = None
    for t in prompt:
        ref = om.step(cache, int(t))
    toks = [oracle.argmax_f32(ref)]
    with bq.Model(cfg, w, max_seq=cap, max_batch=2, flags=bq.LLM_KV_Q8) as m:
        logits = np.empty(cfg["vocab"], np.float32)
        am = np.zeros(1, np.int32)
        m.prefill_batched(1, prompt, logits, am)
        assert m.kv_len(1) == n_prompt
        err = np.abs(logits - ref).max() / np.abs(ref).max()
        assert err <= LOGIT_REL, f"last-token logit error {err:.3e}"
        assert int(am[0]) == toks[0]
        _appended_rows_match(cfg, m, cache, 0, n_prompt, seq=1)
        for _ in range(n):
            toks.append(oracle.argmax_f32(om.step(cache, toks[-1])))
        assert np.array_equal(m.decode_greedy(1, int(am[0]), n), toks[1:])


def test_kv8_refuses_the_paths_that_read_bf16():
    cfg = synth.workload(0)
    w = synth.make_weights(cfg)
    with pytest.raises(bq.LlmError) as e:
        bq.Model(cfg, w, max_seq=16, flags=bq.LLM_KV_Q8 | bq.LLM_MULTI_KERNEL)
    assert e.value.code == -2
