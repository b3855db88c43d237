"""The seeded input generator: determinism and the value recipe of the workloads."""
import numpy as np

import synth


def test_deterministic_and_seed_dependent():
    cfg = synth.workload(0)
    a, b = synth.make_weights(cfg), synth.make_weights(cfg)
    for k in a:
        for f in ("codes", "scales", "mins", "data"):
            if f in a[k]:
                assert np.array_equal(a[k][f], b[k][f])
    c = synth.make_weights(cfg, seed=1)
    assert not np.array_equal(a["L0.wq"]["codes"], c["L0.wq"]["codes"])
    assert np.array_equal(synth.make_prompt(cfg), synth.make_prompt(cfg))


def test_value_recipe():
    cfg = synth.workload(0)
    w = synth.make_weights(cfg)
    t = w["L1.w_up"]
    q = np.concatenate([t["codes"] & 15, t["codes"] >> 4]).ravel()
    counts = np.bincount(q, minlength=16)
    assert counts.min() > 0.8 * q.size / 16 and counts.max() < 1.2 * q.size / 16
    s = t["scales"].astype(np.float64)
    assert s.min() >= 0.002 - 1e-6 and s.max() <= 0.006 + 1e-6
    assert np.array_equal(t["mins"], (-7.5 * s).astype(np.float16))
    e = w["embed"]["data"]
    assert abs(e.std() - 0.02) < 0.001 and e.dtype == np.float32
    nw = w["L0.attn_norm"]["data"]
    assert abs(nw.mean() - 1.0) < 0.005 and abs(nw.std() - 0.01) < 0.003


def test_tied_embedding_is_bf16_and_shapes():
    cfg = synth.workload(2, n_layers=1, vocab=512)
    w = synth.make_weights(cfg)
    assert w["embed"]["kind"] == "bf16" and w["embed"]["data"].shape == (512, 1024)
    assert "lm_head" not in w and w["L0.q_norm"]["data"].shape == (128,)
    assert w["L0.wq"]["codes"].shape == (2048, 512) and w["L0.wo"]["scales"].shape == (1024, 32)


def test_ragged_lengths_and_prefilled_cache():
    cfg = synth.workload(4)
    lens = synth.make_kv_lengths(cfg, 32)
    assert lens.min() >= 512 and lens.max() <= 2048 and len(set(lens.tolist())) > 20
    k, v = synth.make_prefilled_kv(synth.workload(3), 0, 0, 8)
    assert k.shape == (8, 4, 64) and k.dtype == np.uint16
    assert np.array_equal(synth.make_kv_lengths(synth.workload(3), 1), [4096])


def test_weight_byte_model():
    b = synth.weight_bytes(synth.workload(1))
    assert b["codes"] == 517210112 and b["scales_mins"] == 64651264
    b2 = synth.weight_bytes(synth.workload(2))
    assert b2["lm_head_bf16"] == 151936 * 1024 * 2
