"""The checked build (LLMQ_CHECKED=1) on the GPU paths, against the oracle.

Every computed index into a weight stream, a K/V cache row or a partial-sum
array is tested on the device; one outside its buffer would set a status bit
and fail the call. The checked library runs here, in a process of its own,
through the batch-1 persistent step (bf16 and int8 caches), the per-kernel
path, the batched step and batched prefill, on shapes with ragged tails: every
call must succeed and match the oracle at the usual bars.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import numpy as np, torch
import bit_quantized_token_gb300 as bq, oracle, synth
assert bq.CHECKED and bq.LIB_PATH.endswith("libllmq_checked.so")
bq.build(); oracle.build(); torch.cuda.set_device(0)

def greedy(cfg, flags, n=8):
    w = synth.make_weights(cfg); prompt = synth.make_prompt(cfg)
    ref = oracle.greedy_run(oracle.OracleModel(cfg, w), prompt, n, kv="q8" if flags & bq.LLM_KV_Q8 else "bf16")
    with bq.Model(cfg, w, max_seq=len(prompt) + n + 1, flags=flags) as m:
        lg = np.empty(cfg["vocab"], np.float32); am = np.zeros(1, np.int32)
        m.prefill(0, prompt, lg, am)
        err = np.abs(lg - ref["logits"][0]).max() / np.abs(ref["logits"][0]).max()
        toks = [int(am[0])] + list(m.decode_greedy(0, int(am[0]), n))
        m.sync()
    assert err <= 5e-3, (cfg["name"], flags, err)
    # identical greedy tokens, unless the oracle's own top two were within the logit bar there
    for i, (t, r) in enumerate(zip(toks, ref["tokens"])):
        if t != r:
            top2 = np.sort(ref["logits"][i])[-2:]
            assert top2[1] - top2[0] <= 1e-2 * np.abs(ref["logits"][i]).max(), (cfg["name"], flags, i, toks)
            break

tiny = synth.workload(0)
qwen2 = synth.workload(2, n_layers=2, vocab=4099)     # ragged vocabulary tail
for flags in (0, bq.LLM_MULTI_KERNEL, bq.LLM_KV_Q8, bq.LLM_DATAFLOW_STEP):
    greedy(tiny, flags)
greedy(qwen2, 0)
greedy(qwen2, bq.LLM_KV_Q8)

# batched step over ragged caches, and batched prefill of a ragged prompt
cfg = synth.workload(0)
w = synth.make_weights(cfg)
om = oracle.OracleModel(cfg, w)
for kv in ("bf16", "q8"):
    flags = bq.LLM_KV_Q8 if kv == "q8" else 0
    lens = [3, 17, 1, 40]
    with bq.Model(cfg, w, max_seq=48, max_batch=4, flags=flags) as m:
        caches = []
        for b, n in enumerate(lens):
            c = om.new_cache(48, kv=kv)
            for l in range(cfg["n_layers"]):
                k, v = synth.make_prefilled_kv(cfg, l, b, n)
                c.fill(l, k, v); m.kv_write(b, l, 0, k, v)
            c.set_len(n); caches.append(c)
        toks = synth.make_first_tokens(cfg, 4)
        logits = np.empty((4, cfg["vocab"]), np.float32)
        m.decode_step_batch(toks, logits)
        for b in range(4):
            ref = om.step(caches[b], int(toks[b]))
            assert np.abs(logits[b] - ref).max() <= 5e-3 * np.abs(ref).max(), (kv, b)
    with bq.Model(cfg, w, max_seq=80, max_batch=2, flags=flags) as m:
        prompt = synth.make_prompt(cfg, n=45)
        lg = np.empty(cfg["vocab"], np.float32)
        m.prefill_batched(1, prompt, lg)
        c = om.new_cache(80, kv=kv)
        for t in prompt:
            ref = om.step(c, int(t))
        assert np.abs(lg - ref).max() <= 5e-3 * np.abs(ref).max(), kv
print("checked build: every call clean")
"""


def test_checked_build_runs_clean():
    env = dict(os.environ, LLMQ_CHECKED="1", PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-c", SCRIPT], cwd=ROOT, env=env, capture_output=True, text=True, timeout=1500)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "every call clean" in r.stdout
