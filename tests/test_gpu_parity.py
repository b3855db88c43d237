"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Bars (element by element, on the same seeded inputs):
  * 4-bit code unpacking and KV-cache indexing: bit-exact;
  * per-layer hidden states: relative L2 <= 2e-3;
  * logits: max|d| <= 5e-3 * max|logit| at every compared step;
  * greedy tokens identical for the whole run on the three batch-1 workloads.
Kernel-level GEMV checks use a tighter bar derived from fp32 accumulation
(max|d| <= 1e-5 * max|y|, relative L2 <= 2e-6).
"""
import numpy as np
import pytest
import torch

import bit_quantized_token_gb300 as bq
import oracle
from oracle import sampling
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


# ---------------------------------------------------------------- kernel level

@pytest.mark.parametrize("rows,cols", [(3, 64), (5, 128), (7, 5632), (33, 256), (2560, 2048), (2048, 5632),
                                       (1000, 1024), (96, 3072)])
def test_q4_matvec_matches_oracle(rows, cols):
    rng = np.random.default_rng(rows + cols)
    t = synth._q4(rng, rows, cols)
    x = rng.standard_normal(cols).astype(np.float32)
    y = bq.matvec(t, x)
    ref = oracle.matvec(t, x.astype(np.float64))
    assert np.abs(y - ref).max() <= 1e-5 * np.abs(ref).max()
    assert rel_l2(y, ref) <= 2e-6


@pytest.mark.parametrize("rows,cols", [(32, 64), (1000, 1024), (4747, 1024)])
def test_bf16_matvec_matches_dense(rows, cols):
    rng = np.random.default_rng(rows)
    e = synth.bf16_bits_from_f32(rng.normal(0, 0.02, (rows, cols)).astype(np.float32))
    x = rng.standard_normal(cols).astype(np.float32)
    y = bq.matvec(dict(kind="bf16", data=e, rows=rows, cols=cols), x)
    dense = (e.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ref = dense @ x.astype(np.float64)
    assert np.abs(y - ref).max() <= 1e-5 * np.abs(ref).max()


# ---------------------------------------------------------------- bit-exact layout

def _mini(idx, **kw):
    return synth.workload(idx, **kw)


@pytest.mark.parametrize("cfg", [synth.workload(0), synth.workload(2, n_layers=2, vocab=4096)],
                         ids=["tiny", "qwen-shape-2-layers"])
def test_unpack_is_bit_exact(cfg):
    w = synth.make_weights(cfg)
    with bq.Model(cfg, w, max_seq=32) as m:
        for name, t in w.items():
            if t["kind"] != "q4":
                continue
            codes, scales, mins = m.unpack(name, t["rows"], t["cols"])
            assert np.array_equal(codes, t["codes"]), name
            assert np.array_equal(scales, t["scales"].view(np.uint16)), name
            assert np.array_equal(mins, t["mins"].view(np.uint16)), name


def test_kv_write_read_roundtrip_and_append_slot():
    cfg = synth.workload(0)
    w = synth.make_weights(cfg)
    L, H, hd, cap = cfg["n_layers"], cfg["n_kv_heads"], cfg["head_dim"], 24
    with bq.Model(cfg, w, max_seq=cap, max_batch=2) as m:
        # position-coded fill of every slot of sequence 1
        code = lambda l, p: ((np.arange(H * hd, dtype=np.uint16) + 37 * p + 1000 * l) & 0x3FFF).reshape(1, H, hd)
        for l in range(L):
            k = np.concatenate([code(l, p) for p in range(cap)])
            m.kv_write(1, l, 0, k, k ^ 0x4000)
        for l in range(L):
            k, v = m.kv_read(1, l, 0, cap)
            assert np.array_equal(k, np.concatenate([code(l, p) for p in range(cap)]))
            assert np.array_equal(v, k ^ 0x4000)
        # make positions 0..4 the real cache, then append one token at position 5
        m.kv_reset(1)
        prompt = synth.make_prompt(cfg)[:5]
        ref_model = oracle.OracleModel(cfg, w)
        ref_cache = ref_model.new_cache(cap)
        for t in prompt:
            ref_model.step(ref_cache, int(t))
        for l in range(L):
            m.kv_write(1, l, 0, np.transpose(ref_cache.k[l, :, :5], (1, 0, 2)).copy(),
                       np.transpose(ref_cache.v[l, :, :5], (1, 0, 2)).copy())
        assert m.kv_len(1) == 5
        before = [m.kv_read(1, l, 0, cap) for l in range(L)]
        m.decode_step(1, 11)
        ref_model.step(ref_cache, 11)
        assert m.kv_len(1) == 6
        for l in range(L):
            k, v = m.kv_read(1, l, 0, cap)
            # only slot 5 changed, in every layer and head
            assert np.array_equal(k[:5], before[l][0][:5]) and np.array_equal(k[6:], before[l][0][6:])
            assert np.array_equal(v[:5], before[l][1][:5]) and np.array_equal(v[6:], before[l][1][6:])
            # the appended slot holds this token's bf16 K/V (oracle value within one bf16 ulp)
            for got, ref in ((k[5], ref_cache.k[l, :, 5]), (v[5], ref_cache.v[l, :, 5])):
                gf = (got.astype(np.uint32) << 16).view(np.float32)
                rf = (ref.astype(np.uint32) << 16).view(np.float32)
                assert np.all(np.abs(gf - rf) <= np.abs(rf) * 2 ** -7 + 1e-30)
        # sequence 0 was never touched
        assert m.kv_len(0) == 0


# ---------------------------------------------------------------- end to end

def gpu_run(m, cfg, prompt, n_steps, seq=0, hidden=False):
    """prefill(prompt) -> t0, then n_steps decode_step calls feeding back argmax."""
    V = cfg["vocab"]
    logits = np.empty((n_steps + 1, V), np.float32)
    am = np.zeros(1, np.int32)
    hid = []
    m.prefill(seq, prompt, logits[0], am)
    toks = [int(am[0])]
    if hidden:
        hid.append(m.hidden())
    for i in range(n_steps):
        m.decode_step(seq, toks[-1], logits[i + 1], am)
        toks.append(int(am[0]))
        if hidden:
            hid.append(m.hidden())
    return np.array(toks), logits, (np.array(hid) if hidden else None)


def check_against_oracle(cfg, toks, logits, hid, ref, greedy=True):
    if greedy:
        srt = np.sort(ref["logits"], axis=1)
        margins = srt[:, -1] - srt[:, -2]
        mism = np.nonzero(toks != ref["tokens"])[0]
        assert mism.size == 0, (f"greedy token mismatch at steps {mism[:5]}, oracle margin there "
                                f"{margins[mism[:5]]}, gpu tokens {toks[mism[:5]]} vs {ref['tokens'][mism[:5]]}")
    err = np.abs(logits - ref["logits"]).max(axis=1) / np.abs(ref["logits"]).max(axis=1)
    assert err.max() <= LOGIT_REL, f"logit error {err.max():.3e} at step {err.argmax()}"
    if hid is not None:
        for s in range(hid.shape[0]):
            for l in range(hid.shape[1]):
                r = rel_l2(hid[s, l], ref["hidden"][s, l])
                assert r <= HIDDEN_RL2, f"hidden rel L2 {r:.3e} at step {s} layer {l}"
    return err.max()


@pytest.mark.parametrize("flags", [0, bq.LLM_NO_GRAPH, bq.LLM_MULTI_KERNEL, bq.LLM_MULTI_KERNEL | bq.LLM_NO_GRAPH,
                                   bq.LLM_MULTI_KERNEL | bq.LLM_NO_PDL, bq.LLM_DATAFLOW_STEP],
                         ids=["persistent", "persistent-eager", "multi-kernel-graph+pdl", "multi-kernel-eager+pdl",
                              "multi-kernel-graph", "dataflow"])
def test_tiny_llama_greedy_matches_oracle(flags):
    cfg = synth.workload(0)
    w = synth.make_weights(cfg)
    prompt = synth.make_prompt(cfg)
    n = cfg["decode_steps"]
    ref = oracle.greedy_run(oracle.OracleModel(cfg, w), prompt, n, hidden=True)
    with bq.Model(cfg, w, max_seq=64, max_batch=2, flags=flags) as m:
        toks, logits, hid = gpu_run(m, cfg, prompt, n, seq=1, hidden=True)
        check_against_oracle(cfg, toks, logits, hid, ref)
        # the device-fed greedy loop gives the same tokens
        m.kv_reset(1)
        am = np.zeros(1, np.int32)
        m.prefill(1, prompt, None, am)
        assert int(am[0]) == ref["tokens"][0]
        assert np.array_equal(m.decode_greedy(1, int(am[0]), n), ref["tokens"][1:])


def test_bit_reproducible():
    cfg = synth.workload(0)
    w = synth.make_weights(cfg)
    prompt = synth.make_prompt(cfg)
    outs = []
    for _ in range(2):
        with bq.Model(cfg, w, max_seq=64) as m:
            outs.append(gpu_run(m, cfg, prompt, 6)[1])
    assert np.array_equal(outs[0], outs[1])


@pytest.mark.parametrize("flags", [0, bq.LLM_DATAFLOW_STEP], ids=["barrier", "dataflow"])
def test_qwen_shape_two_layers_full_vocab(flags):
    # tied bf16 LM head over the full 151936-token vocabulary, q/k norm, NEOX
    cfg = synth.workload(2, n_layers=2)
    w = synth.make_weights(cfg)
    prompt = synth.make_prompt(cfg)
    ref = oracle.greedy_run(oracle.OracleModel(cfg, w), prompt, 20, hidden=True)
    with bq.Model(cfg, w, max_seq=64, flags=flags) as m:
        toks, logits, hid = gpu_run(m, cfg, prompt, 20, hidden=True)
        if flags:
            assert m.stats()["kernels_per_step"] == 1
    check_against_oracle(cfg, toks, logits, hid, ref)


@pytest.mark.parametrize("idx", [1, 2], ids=["tinyllama-1.1b", "qwen3-0.6b"])
def test_full_size_greedy_matches_oracle(idx):
    cfg = synth.workload(idx)
    w = synth.make_weights(cfg)
    prompt = synth.make_prompt(cfg)
    n = cfg["decode_steps"]
    ref = oracle.greedy_run(oracle.OracleModel(cfg, w), prompt, n, hidden=True)
    for flags in (0, bq.LLM_MULTI_KERNEL, bq.LLM_DATAFLOW_STEP):
        with bq.Model(cfg, w, max_seq=len(prompt) + n + 1, flags=flags) as m:
            toks, logits, hid = gpu_run(m, cfg, prompt, n, hidden=True)
        check_against_oracle(cfg, toks, logits, hid, ref)


def test_long_context_teacher_forced():
    # 4096 pre-filled positions of N(0,1) bf16 K/V, then 64 steps fed with the
    # oracle's greedy tokens; logits compared at every step
    cfg = synth.workload(3)
    w = synth.make_weights(cfg)
    n_pre, n = cfg["prefill_kv"], cfg["decode_steps"]
    cap = n_pre + n + 1
    om = oracle.OracleModel(cfg, w)
    cache = om.new_cache(cap)
    with bq.Model(cfg, w, max_seq=cap) as m:
        for l in range(cfg["n_layers"]):
            k, v = synth.make_prefilled_kv(cfg, l, 0, n_pre)
            cache.fill(l, k, v)
            m.kv_write(0, l, 0, k, v)
        cache.set_len(n_pre)
        tok = int(synth.make_first_tokens(cfg, 1)[0])
        logits = np.empty(cfg["vocab"], np.float32)
        worst = 0.0
        for i in range(n):
            ref, ref_h = om.step(cache, tok, hidden=True)
            m.decode_step(0, tok, logits)
            err = np.abs(logits - ref).max() / np.abs(ref).max()
            worst = max(worst, err)
            assert err <= LOGIT_REL, f"step {i}: logit error {err:.3e}"
            hid = m.hidden()
            for l in range(cfg["n_layers"] + 1):
                assert rel_l2(hid[l], ref_h[l]) <= HIDDEN_RL2
            tok = oracle.argmax_f32(ref)
        assert m.kv_len(0) == n_pre + n


@pytest.mark.parametrize("cfg,n_pre", [(synth.workload(1, n_layers=2, vocab=4096), 500),
                                       (synth.workload(2, n_layers=2, vocab=4096), 370)],
                         ids=["tinyllama-shape-fused-then-split", "qwen3-shape-split"])
@pytest.mark.parametrize("flags", [0, bq.LLM_DATAFLOW_STEP], ids=["barrier", "dataflow"])
def test_attention_paths_across_the_switch(cfg, n_pre, flags):
    # Short caches, one kv head per o-projection range (the TinyLlama shape):
    # every CTA of the persistent step attends over the cache inside the
    # o-projection's input build; from 4 passes of positions (512) on, the
    # step variant with a separate attention phase does it. Teacher-forced
    # steps across that length compare both (and the append in each) with the
    # oracle; the Qwen3 shape (two kv heads per range) always splits.
    w = synth.make_weights(cfg)
    n = 24
    cap = n_pre + n + 1
    om = oracle.OracleModel(cfg, w)
    cache = om.new_cache(cap)
    with bq.Model(cfg, w, max_seq=cap, flags=flags) as m:
        for l in range(cfg["n_layers"]):
            k, v = synth.make_prefilled_kv(cfg, l, 0, n_pre)
            cache.fill(l, k, v)
            m.kv_write(0, l, 0, k, v)
        cache.set_len(n_pre)
        tok = int(synth.make_first_tokens(cfg, 1)[0])
        logits = np.empty(cfg["vocab"], np.float32)
        for i in range(n):
            ref, ref_h = om.step(cache, tok, hidden=True)
            m.decode_step(0, tok, logits)
            err = np.abs(logits - ref).max() / np.abs(ref).max()
            assert err <= LOGIT_REL, f"step {i} (cache length {n_pre + i + 1}): logit error {err:.3e}"
            hid = m.hidden()
            for l in range(cfg["n_layers"] + 1):
                assert rel_l2(hid[l], ref_h[l]) <= HIDDEN_RL2, f"step {i} layer {l}"
            tok = oracle.argmax_f32(ref)
        assert m.kv_len(0) == n_pre + n
        for l in range(cfg["n_layers"]):
            k, v = m.kv_read(0, l, 0, n_pre + n)
            for name, got, rc in (("K", k[n_pre:], cache.k[l, :, n_pre:n_pre + n]),
                                  ("V", v[n_pre:], cache.v[l, :, n_pre:n_pre + n])):
                gf = (got.astype(np.uint32) << 16).view(np.float32)
                rf = (np.transpose(rc, (1, 0, 2)).astype(np.uint32) << 16).view(np.float32)
                # one bf16 ulp of the oracle's value, or, where the element is a
                # near-cancellation, the absolute error the layer's fp32 input
                # carries into it (2^-16 of the head vector's largest element;
                # the hidden states themselves are held to rel. L2 2e-3 above)
                tol = np.maximum(np.abs(rf) * 2 ** -7, np.abs(rf).max(axis=2, keepdims=True) * 2 ** -16)
                bad = np.argwhere(~(np.abs(gf - rf) <= tol))
                assert bad.size == 0, (f"appended {name} of layer {l}: {len(bad)} elements off, first (step, head, dim) "
                                       f"{bad[:4].tolist()}, gpu {[float(gf[tuple(b)]) for b in bad[:4]]}, "
                                       f"oracle {[float(rf[tuple(b)]) for b in bad[:4]]}")


@pytest.mark.parametrize("cfg,n_prompt", [(synth.workload(0), 70), (synth.workload(2, n_layers=2, vocab=4096), 45),
                                          (synth.workload(1), 40)],
                         ids=["tiny-3-chunks", "qwen3-shape-2-chunks", "tinyllama-1.1b-2-chunks"])
def test_batched_prefill_matches_token_by_token(cfg, n_prompt):
    # Batched prompt processing (chunks of up to 32 tokens through the batched
    # pipeline) against the oracle's token-by-token prefill: last logits,
    # greedy token, every appended K/V row; then greedy decoding continues
    # from that cache with the oracle's tokens.
    w = synth.make_weights(cfg)
    prompt = synth.make_prompt(cfg, n=n_prompt)
    n = 8
    ref = oracle.greedy_run(oracle.OracleModel(cfg, w), prompt, n)
    cap = n_prompt + n + 1
    om = oracle.OracleModel(cfg, w)
    cache = om.new_cache(cap)
    for t in prompt:
        om.step(cache, int(t))
    with bq.Model(cfg, w, max_seq=cap, max_batch=2) as m:
        logits = np.empty(cfg["vocab"], np.float32)
        am = np.zeros(1, np.int32)
        m.prefill_batched(1, prompt, logits, am)
        assert m.kv_len(1) == n_prompt and m.kv_len(0) == 0
        err = np.abs(logits - ref["logits"][0]).max() / np.abs(ref["logits"][0]).max()
        assert err <= LOGIT_REL, f"last-token logit error {err:.3e}"
        assert int(am[0]) == ref["tokens"][0] == int(np.argmax(logits))
        for l in range(cfg["n_layers"]):
            k, v = m.kv_read(1, l, 0, n_prompt)
            for name, got, rc in (("K", k, cache.k[l, :, :n_prompt]), ("V", v, cache.v[l, :, :n_prompt])):
                gf = (got.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
                rf = (np.transpose(rc, (1, 0, 2)).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
                # K/V are bf16-rounded projections: where the GPU's fp32 and the
                # oracle's fp64 values round to different bf16 neighbours (2^-8
                # relative) the difference travels through the later layers'
                # attention, so each layer's appended K (V) is held to the hidden
                # state's bound (rel. L2 2e-3); every (position, head) vector
                # within 1e-2 still catches a wrong position, head or chunk row
                tot = np.linalg.norm(gf - rf) / np.linalg.norm(rf)
                assert tot <= HIDDEN_RL2, f"{name} of layer {l}: rel. L2 {tot:.2e}"
                rl2 = np.linalg.norm(gf - rf, axis=2) / np.linalg.norm(rf, axis=2)
                assert rl2.max() <= 1e-2, (f"{name} of layer {l}: rel. L2 {rl2.max():.2e} at (pos, head) "
                                           f"{np.unravel_index(rl2.argmax(), rl2.shape)}")
        assert np.array_equal(m.decode_greedy(1, int(am[0]), n), ref["tokens"][1:])


# ---------------------------------------------------------------- sampled choice

def _sampled_matches(logits, token, T, k, p, seed, seq, pos):
    """The oracle's choice from the same fp32 logits and draw; a decision may
    differ only where its target lies within rounding of a cumulative boundary."""
    ref, info = sampling.sample(logits, T, k, p, sampling.uniform(seed, seq, pos))
    if token == ref:
        return True
    c, n = info["cum"], info["n"]
    near = min(abs(c[j] - info["target"]) for j in range(n)) < 1e-5 or abs(c[n - 1] - p) < 1e-5
    assert near and token in info["ids"][:n], (f"position {pos}: sampled {token}, oracle {ref} "
                                               f"(target {info['target']:.6f}, cumulative {c[:n]})")
    return False


@pytest.mark.parametrize("idx,flags", [(0, 0), (0, bq.LLM_MULTI_KERNEL), (1, 0)],
                         ids=["tiny-persistent", "tiny-multi-kernel", "tinyllama-1.1b"])
def test_sampled_choice_matches_the_oracle(idx, flags):
    # temperature / top-k / top-p with the Philox draw of (seed, sequence,
    # position): every chosen token equals the oracle's choice from the GPU's
    # own logits; the device-fed loop reproduces them from the seed alone
    cfg = synth.workload(idx)
    w = synth.make_weights(cfg)
    prompt = synth.make_prompt(cfg)
    T, k, p, seed, seq, n = 0.9, 40, 0.95, 20261202, 1, 24
    with bq.Model(cfg, w, max_seq=len(prompt) + n + 2, max_batch=2, flags=flags) as m:
        m.set_sampling(T, k, p, seed)
        logits = np.empty(cfg["vocab"], np.float32)
        am = np.zeros(1, np.int32)
        m.prefill(seq, prompt, logits, am)
        pos = len(prompt) - 1
        toks = [int(am[0])]
        exact = [_sampled_matches(logits, toks[-1], T, k, p, seed, seq, pos)]
        not_greedy = [toks[-1] != int(np.argmax(logits))]
        for _ in range(n):
            pos += 1
            m.decode_step(seq, toks[-1], logits, am)
            toks.append(int(am[0]))
            exact.append(_sampled_matches(logits, toks[-1], T, k, p, seed, seq, pos))
            not_greedy.append(toks[-1] != int(np.argmax(logits)))
        assert sum(exact) >= len(exact) - 1 and any(not_greedy)
        # the device-fed loop draws the same tokens from the same seed
        m.kv_reset(seq)
        m.prefill(seq, prompt, None, am)
        assert int(am[0]) == toks[0]
        assert list(m.decode_greedy(seq, toks[0], n)) == toks[1:]
        # batched prompt processing samples the same first token
        m.kv_reset(seq)
        m.prefill_batched(seq, prompt, logits, am)
        _sampled_matches(logits, int(am[0]), T, k, p, seed, seq, len(prompt) - 1)
        # temperature 0: greedy again
        m.set_sampling(0.0)
        m.kv_reset(seq)
        m.prefill(seq, prompt, logits, am)
        assert int(am[0]) == int(np.argmax(logits))
        with pytest.raises(bq.LlmError):
            m.set_sampling(0.5, 0)


# ---------------------------------------------------------------- errors

def test_error_paths_leave_model_usable():
    cfg = synth.workload(0)
    w = synth.make_weights(cfg)
    with bq.Model(cfg, w, max_seq=4) as m:
        with pytest.raises(bq.LlmError) as e:
            m.decode_step(0, cfg["vocab"])
        assert e.value.code == -1
        with pytest.raises(bq.LlmError) as e:
            m.prefill(0, [1, 2, 3, 4, 5])
        assert e.value.code == -4
        m.prefill(0, [1, 2, 3])
        m.decode_step(0, 4)
        with pytest.raises(bq.LlmError) as e:
            m.decode_step(0, 5)
        assert e.value.code == -4
        m.kv_reset(0)
        m.decode_step(0, 5)
    bad = dict(cfg, head_dim=96)
    with pytest.raises(bq.LlmError) as e:
        bq.Model(bad, w, max_seq=8)
    assert e.value.code == -2 and "head_dim" in str(e.value)
    w2 = dict(w)
    del w2["L1.wo"]
    with pytest.raises(bq.LlmError) as e:
        bq.Model(cfg, w2, max_seq=8)
    assert e.value.code == -8 and "L1.wo" in str(e.value)


# ---------------------------------------------------------------- batched decode

def _batched_vs_oracle(cfg, lens, n_steps, seed_tokens, hidden=False, kv8=False):
    """Ragged pre-filled caches, teacher-forced batched steps compared per sequence.

    Every step: logits at 5e-3 * max|logit|; the greedy choice equal to the
    oracle's (a different choice passes only where the oracle's own top two
    logits lie within twice that bar of each other, and is then a top logit
    of the oracle too); with `hidden`, every layer's residual at rel. L2 2e-3.
    """
    B = len(lens)
    w = synth.make_weights(cfg)
    om = oracle.OracleModel(cfg, w)
    cap = int(max(lens)) + n_steps + 1
    caches = []
    flags = (bq.LLM_DEBUG_BATCH_HIDDEN if hidden else 0) | (bq.LLM_KV_Q8 if kv8 else 0)
    near_ties = 0
    with bq.Model(cfg, w, max_seq=cap, max_batch=B, flags=flags) as m:
        for b in range(B):
            c = om.new_cache(int(lens[b]) + n_steps + 1, kv="q8" if kv8 else "bf16")
            for l in range(cfg["n_layers"]):
                k, v = synth.make_prefilled_kv(cfg, l, b, int(lens[b]))
                c.fill(l, k, v)
                m.kv_write(b, l, 0, k, v)
            c.set_len(int(lens[b]))
            caches.append(c)
        toks = np.array(seed_tokens, np.int32)
        logits = np.empty((B, cfg["vocab"]), np.float32)
        am = np.zeros(B, np.int32)
        worst = 0.0
        for s in range(n_steps):
            m.decode_step_batch(toks, logits, am)
            hid = m.hidden_batch() if hidden else None
            nxt = np.empty(B, np.int32)
            for b in range(B):
                if hidden:
                    ref, ref_h = om.step(caches[b], int(toks[b]), hidden=True)
                    for l in range(cfg["n_layers"] + 1):
                        r = rel_l2(hid[l, b], ref_h[l])
                        assert r <= HIDDEN_RL2, f"step {s} seq {b} layer {l}: hidden rel L2 {r:.3e}"
                else:
                    ref = om.step(caches[b], int(toks[b]))
                scale = np.abs(ref).max()
                err = np.abs(logits[b] - ref).max() / scale
                worst = max(worst, err)
                assert err <= LOGIT_REL, f"step {s} seq {b}: logit error {err:.3e}"
                choice = oracle.argmax_f32(ref)
                if int(am[b]) != choice:
                    top2 = np.sort(ref)[-2:]
                    assert top2[1] - top2[0] <= 2 * LOGIT_REL * scale, (
                        f"step {s} seq {b}: greedy choice {int(am[b])}, oracle {choice} by a margin "
                        f"{(top2[1] - top2[0]) / scale:.3e} of max|logit|")
                    assert ref[int(am[b])] >= top2[0], f"step {s} seq {b}: choice outside the oracle's top two"
                    near_ties += 1
                nxt[b] = choice
            toks = nxt
        for b in range(B):
            assert m.kv_len(b) == int(lens[b]) + n_steps
    assert near_ties <= max(1, B * n_steps // 100)
    return worst


def test_batched_tiny_matches_oracle():
    cfg = synth.workload(0)
    lens = [3, 17, 1, 40]
    _batched_vs_oracle(cfg, lens, 6, synth.make_first_tokens(cfg, 4), hidden=True)


def test_batched_qwen_shape_ragged_two_layers():
    # 32 sequences, cache lengths uniform in [512, 2048], full 151936-token vocabulary
    cfg = synth.workload(4, n_layers=2)
    lens = synth.make_kv_lengths(cfg, 32)
    _batched_vs_oracle(cfg, lens, 3, synth.make_first_tokens(cfg, 32), hidden=True)


def test_batched_tied_head_ragged_vocabulary():
    # the tied bf16 LM head with a vocabulary that is not a multiple of 32
    # rows (126 row tiles over the persistent head's CTAs, the last tile
    # partly masked), 3 sequences (29 padding token rows), caches of 1..3 passes
    cfg = synth.workload(2, n_layers=1, vocab=4001)
    _batched_vs_oracle(cfg, [70, 130, 5], 3, synth.make_first_tokens(cfg, 3), hidden=True)


def test_batched_tied_head_wider_than_the_resident_input():
    # a tied bf16 head of dim 2048: its staged 32-token input (2 x 32 x 2056
    # bf16) does not fit in one CTA's shared memory beside the ring, so the
    # LM head runs as the split-K GEMV with the greedy epilogue instead
    cfg = synth.workload(2, n_layers=1, vocab=4096, dim=2048)
    _batched_vs_oracle(cfg, [40, 300, 7], 3, synth.make_first_tokens(cfg, 3), hidden=True)


def test_batched_tiny_int8_kv_matches_oracle():
    # the grouped int8 cache (LLM_KV_Q8) against the oracle's int8 caches
    cfg = synth.workload(0)
    _batched_vs_oracle(cfg, [3, 17, 1, 40], 6, synth.make_first_tokens(cfg, 4), hidden=True, kv8=True)


def test_batched_workload_full_size_int8_kv():
    cfg = synth.workload(4)
    lens = synth.make_kv_lengths(cfg, 32)
    _batched_vs_oracle(cfg, lens, 16, synth.make_first_tokens(cfg, 32), hidden=True, kv8=True)


def test_batched_workload_full_size():
    # the full batched workload: 32 sequences of the Qwen3-0.6B shape, caches
    # of 512..2048 positions, all 64 decode steps teacher-forced with every
    # layer's residual of every sequence checked
    cfg = synth.workload(4)
    lens = synth.make_kv_lengths(cfg, 32)
    _batched_vs_oracle(cfg, lens, cfg["decode_steps"], synth.make_first_tokens(cfg, 32), hidden=True)
