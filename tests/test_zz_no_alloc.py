"""The matvec entry point that allocates no device memory.

It serves callers that cannot call cudaMalloc where they call it (their
device memory belongs to a pool reserved at start-up, or their loop cannot
afford the stall of cudaMalloc/cudaFree). Its scratch lives in a static
device array inside the library. Here its result is checked against the
oracle's fp64 matvec on two calls in a row (every call reuses the array the
previous call left behind), after other models and calls have set the GEMV
kernel's shared-memory limit for smaller matrices, on a non-default stream,
on a capturing stream (refused), past its scratch size (refused, the model
stays usable), and for device memory left unchanged. This file is collected
last so that a failure here does not stop the rest of the GPU suite.
"""
import numpy as np
import pytest
import torch

import bit_quantized_token_gb300 as bq
import oracle
import synth

pytestmark = pytest.mark.gpu

INVALID_ARG, UNSUPPORTED, NOT_FOUND = -1, -2, -8


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available()
    bq.build()
    oracle.build()


def _reference(t, x):
    if t.get("kind") == "bf16":
        dense = (np.asarray(t["data"]).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        return dense @ x.astype(np.float64)
    return oracle.matvec(t, x.astype(np.float64))


def _check_calls(m, name, t, n_calls=2, stream=None):
    for call in range(n_calls):
        g = torch.Generator().manual_seed(100 * call + int(t["rows"]))
        x = torch.randn(int(t["cols"]), generator=g).cuda()
        y = torch.full((int(t["rows"]),), float("nan"), device="cuda")
        torch.cuda.synchronize()
        bq.matvec_noalloc(m, name, x, y, stream=stream)
        got = y.cpu().numpy()
        ref = _reference(t, x.cpu().numpy())
        # the bar of the kernel-level GEMV parity tests (fp32 accumulation)
        assert np.abs(got - ref).max() <= 1e-5 * np.abs(ref).max(), (name, call)


@pytest.mark.parametrize("name", ["L1.w_down", "L0.wk", "lm_head"])
def test_noalloc_matvec_matches_oracle(name):
    cfg = synth.workload(0)
    w = synth.make_weights(cfg)
    with bq.Model(cfg, w, max_seq=16) as m:
        _check_calls(m, name, w[name])


def test_noalloc_matvec_tied_bf16_lm_head():
    cfg = synth.workload(2, n_layers=1, vocab=20000)
    w = synth.make_weights(cfg)
    with bq.Model(cfg, w, max_seq=16) as m:
        _check_calls(m, "embed", w["embed"])
        with pytest.raises(bq.LlmError) as e:
            bq.matvec_noalloc(m, "L0.w_gate", torch.zeros(1024, device="cuda"), torch.zeros(3072, device="cuda"))
        assert e.value.code == NOT_FOUND


def test_noalloc_after_smaller_models_and_calls():
    # The GEMV kernel's shared-memory limit is process-wide: a model with a
    # 5632-wide down projection, then a model whose widest input is 768, then
    # a kernel-level matvec on a 64-wide matrix; the first model's w_down
    # (K = 5632, well over the 48 KB default) must still run.
    big_cfg = synth.workload(1, n_layers=1, vocab=4096)
    big_w = synth.make_weights(big_cfg)
    with bq.Model(big_cfg, big_w, max_seq=16) as big:
        small_cfg = synth.workload(0)
        with bq.Model(small_cfg, synth.make_weights(small_cfg), max_seq=16):
            pass
        rng = np.random.default_rng(5)
        bq.matvec(synth._q4(rng, 3, 64), rng.standard_normal(64).astype(np.float32))
        _check_calls(big, "L0.w_down", big_w["L0.w_down"], n_calls=1)


def test_noalloc_on_a_torch_stream_and_memory_unchanged():
    cfg = synth.workload(0)
    w = synth.make_weights(cfg)
    with bq.Model(cfg, w, max_seq=16) as m:
        s = torch.cuda.Stream()
        _check_calls(m, "L1.w_down", w["L1.w_down"], stream=s.cuda_stream)
        t = w["L0.wq"]
        x = torch.randn(int(t["cols"]), device="cuda")
        y = torch.empty(int(t["rows"]), device="cuda")
        bq.matvec_noalloc(m, "L0.wq", x, y, stream=s.cuda_stream)  # warm
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        for _ in range(5):
            bq.matvec_noalloc(m, "L0.wq", x, y, stream=s.cuda_stream)
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free0


def test_noalloc_refuses_a_capturing_stream_without_poisoning():
    cfg = synth.workload(0)
    w = synth.make_weights(cfg)
    with bq.Model(cfg, w, max_seq=16) as m:
        t = w["L0.wk"]
        x = torch.randn(int(t["cols"]), device="cuda")
        y = torch.empty(int(t["rows"]), device="cuda")
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        raised = None
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            try:
                bq.matvec_noalloc(m, "L0.wk", x, y, stream=s.cuda_stream)
            except bq.LlmError as e:
                raised = e
        assert raised is not None and raised.code == INVALID_ARG
        _check_calls(m, "L0.wk", t, n_calls=1)
        logits = np.empty(cfg["vocab"], np.float32)
        m.decode_step(0, 1, logits)
        assert np.isfinite(logits).all()


def test_noalloc_refuses_a_matrix_beyond_its_scratch():
    # A 4-bit LM head of 600000 rows over 256 inputs: two CTAs share each
    # 32-row tile, so it needs 18750 x 2 x 32 partial floats, beyond the
    # 2^20 the static array holds. The call is refused; the model decodes.
    cfg = synth.workload(0, n_layers=1, vocab=600000)
    w = synth.make_weights(cfg)
    with bq.Model(cfg, w, max_seq=16) as m:
        x = torch.randn(cfg["dim"], device="cuda")
        y = torch.empty(cfg["vocab"], device="cuda")
        with pytest.raises(bq.LlmError) as e:
            bq.matvec_noalloc(m, "lm_head", x, y)
        assert e.value.code == UNSUPPORTED
        logits = np.empty(cfg["vocab"], np.float32)
        m.decode_step(0, 7, logits)
        assert np.isfinite(logits).all()
        _check_calls(m, "L0.w_down", w["L0.w_down"], n_calls=1)
