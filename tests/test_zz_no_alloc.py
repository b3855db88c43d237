"""The matvec entry point that allocates no device memory.

It serves callers that cannot call cudaMalloc where they call it (their
device memory belongs to a pool reserved at start-up, or their loop cannot
afford the stall of cudaMalloc/cudaFree). Its scratch lives in a static
device array inside the library. Here its result is checked against the
allocating entry point (llm_op_matvec) on the same weights, on two calls in a
row, because every call reuses the array the previous call left behind.
This file is collected last so that a failure here does not stop the rest of
the GPU suite.
"""
import numpy as np
import pytest
import torch

import bit_quantized_token_gb300 as bq
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available()
    bq.build()


def _check_two_calls(m, name, t):
    for call in range(2):
        g = torch.Generator().manual_seed(100 * call + t["rows"])
        x = torch.randn(t["cols"], generator=g).cuda()
        y = torch.full((t["rows"],), float("nan"), device="cuda")
        bq.matvec_noalloc(m, name, x, y)
        got = y.cpu().numpy()
        ref = bq.matvec(t, x.cpu().numpy())
        # the same bar as the kernel-level GEMV parity tests
        assert np.abs(got - ref).max() <= 1e-5 * np.abs(ref).max(), (name, call)


@pytest.mark.parametrize("name", ["L1.w_down", "L0.wk", "lm_head"])
def test_noalloc_matvec_matches_allocating_entry_point(name):
    cfg = synth.workload(0)
    w = synth.make_weights(cfg)
    with bq.Model(cfg, w, max_seq=16) as m:
        _check_two_calls(m, name, w[name])


def test_noalloc_matvec_tied_bf16_lm_head():
    cfg = synth.workload(2, n_layers=1, vocab=20000)
    w = synth.make_weights(cfg)
    with bq.Model(cfg, w, max_seq=16) as m:
        _check_two_calls(m, "embed", w["embed"])
        with pytest.raises(bq.LlmError) as e:
            bq.matvec_noalloc(m, "L0.w_gate", torch.zeros(1024, device="cuda"), torch.zeros(3072, device="cuda"))
        assert e.value.code == -8
