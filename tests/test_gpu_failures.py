"""Failure paths of the decode step, made on the host or by a bounded wait.

Nothing here faults, traps or hangs the GPU:
  * TIMEOUT: a test-only model flag makes every grid barrier of the persistent
    step wait for one arrival more than its CTAs make, with a 1 ms limit. The
    first barrier's wait runs out, the kernel sets its status word and every
    CTA returns; the call reports LLM_ERR_TIMEOUT and poisons the model. A
    fresh model on the same GPU then decodes like the oracle.
  * NAN: a NaN planted on the host in the final norm weight makes every logit
    NaN; the logit reduction reports LLM_ERR_NAN.
  * OOM: a host hook makes one device allocation of llm_model_create fail;
    create returns LLM_ERR_OOM naming the buffer and frees what it took.
"""
import numpy as np
import pytest
import torch

import bit_quantized_token_gb300 as bq
import oracle
import synth

pytestmark = pytest.mark.gpu

OOM, TIMEOUT, NAN = -3, -6, -7


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available()
    bq.build()
    oracle.build()


def _fresh_model_matches_oracle(cfg, w, n=4):
    prompt = synth.make_prompt(cfg)
    ref = oracle.greedy_run(oracle.OracleModel(cfg, w), prompt, n)
    with bq.Model(cfg, w, max_seq=64) as m:
        am = np.zeros(1, np.int32)
        m.prefill(0, prompt, None, am)
        toks = [int(am[0])] + list(m.decode_greedy(0, int(am[0]), n))
    assert toks == list(ref["tokens"])


def test_expired_wait_returns_timeout_and_poisons():
    cfg = synth.workload(0)
    w = synth.make_weights(cfg)
    logits = np.empty(cfg["vocab"], np.float32)
    with bq.Model(cfg, w, max_seq=64, flags=bq.LLM_TEST_EXPIRE_WAIT) as m:
        assert m.stats()["kernels_per_step"] == 1  # the persistent step serves the call
        with pytest.raises(bq.LlmError) as e:
            m.decode_step(0, 3, logits)
        assert e.value.code == TIMEOUT
        # poisoned: later calls report the same status without launching
        with pytest.raises(bq.LlmError) as e:
            m.decode_step(0, 3, logits)
        assert e.value.code == TIMEOUT
    torch.cuda.synchronize()  # the context is intact
    _fresh_model_matches_oracle(cfg, w)


def test_nan_norm_weight_returns_nan():
    cfg = synth.workload(0)
    w = synth.make_weights(cfg)
    bad = dict(w["final_norm"])
    bad["data"] = bad["data"].copy()
    bad["data"][5] = np.nan
    w_bad = dict(w, final_norm=bad)
    logits = np.empty(cfg["vocab"], np.float32)
    for flags in (0, bq.LLM_MULTI_KERNEL):
        with bq.Model(cfg, w_bad, max_seq=64, flags=flags) as m:
            with pytest.raises(bq.LlmError) as e:
                m.decode_step(0, 3, logits)
            assert e.value.code == NAN
            assert np.isnan(logits).all()
            # not poisoning: the next call runs (and finds the same NaN)
            with pytest.raises(bq.LlmError) as e:
                m.decode_step(0, 4, logits)
            assert e.value.code == NAN
    _fresh_model_matches_oracle(cfg, w)


@pytest.mark.parametrize("nth", [1, 5])
def test_failed_allocation_returns_oom(nth):
    cfg = synth.workload(1, n_layers=2, vocab=4096)
    w = synth.make_weights(cfg)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    bq.debug_fail_alloc(nth)
    try:
        with pytest.raises(bq.LlmError) as e:
            bq.Model(cfg, w, max_seq=64)
    finally:
        bq.debug_fail_alloc(0)
    assert e.value.code == OOM
    assert "device allocation failed" in str(e.value)
    torch.cuda.synchronize()
    # what create had allocated is back (the weights alone are ~50 MB)
    assert torch.cuda.mem_get_info()[0] >= free0 - (8 << 20)
    _fresh_model_matches_oracle(synth.workload(0), synth.make_weights(synth.workload(0)))
