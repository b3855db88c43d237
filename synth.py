"""Seeded synthetic inputs for the 4-bit decode step.

This module only draws random numbers and lays them out in the canonical
packed format that both the CUDA library and the CPU oracle consume. It holds
none of the decoder's arithmetic: no dequantisation, no matvec, no norm, no
RoPE, no attention. Values that the method itself rounds (the bf16 KV cache,
the fp32 logits) are never produced here.

Canonical 4-bit linear ``[out, in]`` (group size 64 along ``in``):

* ``codes``  uint8  ``[out][in/2]`` -- element ``2j`` in the low nibble of byte
  ``j``, element ``2j+1`` in the high nibble;
* ``scales`` fp16   ``[out][in/64]``;
* ``mins``   fp16   ``[out][in/64]``;

so that ``w[r][c] = scale[r][c//64] * q + min[r][c//64]`` with ``q`` the code.

Value recipe (per workload): codes uniform over 0..15, ``scale`` = fp16 of
U(0.002, 0.006), ``min`` = fp16 of ``-7.5 * scale``; norm weights fp32 of
1 + N(0, 0.01); embeddings fp32 N(0, 0.02), or bf16 (round to nearest even)
N(0, 0.02) when the embedding doubles as the LM head; prompts uniform over the
vocabulary; pre-filled KV caches bf16 N(0, 1).
"""
from __future__ import annotations

import numpy as np

GROUP = 64

# Workload shapes. Index = workload number used throughout the tests/bench.
WORKLOADS = {
    0: dict(name="tiny-llama", dim=256, n_layers=4, n_heads=4, n_kv_heads=2, head_dim=64,
            ffn_dim=768, vocab=2048, norm_eps=1e-5, rope_theta=1e4, rope_neox=0, qk_norm=0,
            tied=0, prompt_len=16, decode_steps=16, batch=1, prefill_kv=0),
    1: dict(name="tinyllama-1.1b", dim=2048, n_layers=22, n_heads=32, n_kv_heads=4, head_dim=64,
            ffn_dim=5632, vocab=32000, norm_eps=1e-5, rope_theta=1e4, rope_neox=0, qk_norm=0,
            tied=0, prompt_len=6, decode_steps=128, batch=1, prefill_kv=0),
    2: dict(name="qwen3-0.6b", dim=1024, n_layers=28, n_heads=16, n_kv_heads=8, head_dim=128,
            ffn_dim=3072, vocab=151936, norm_eps=1e-5, rope_theta=1e6, rope_neox=1, qk_norm=1,
            tied=1, prompt_len=17, decode_steps=256, batch=1, prefill_kv=0),
    3: dict(name="tinyllama-1.1b-kv4096", dim=2048, n_layers=22, n_heads=32, n_kv_heads=4,
            head_dim=64, ffn_dim=5632, vocab=32000, norm_eps=1e-5, rope_theta=1e4, rope_neox=0,
            qk_norm=0, tied=0, prompt_len=0, decode_steps=64, batch=1, prefill_kv=4096),
    4: dict(name="qwen3-0.6b-batch32", dim=1024, n_layers=28, n_heads=16, n_kv_heads=8,
            head_dim=128, ffn_dim=3072, vocab=151936, norm_eps=1e-5, rope_theta=1e6, rope_neox=1,
            qk_norm=1, tied=1, prompt_len=0, decode_steps=64, batch=32, prefill_kv=-1,
            kv_len_lo=512, kv_len_hi=2048),
}

BASE_SEED = 20260


def workload(idx: int, **overrides) -> dict:
    cfg = dict(WORKLOADS[idx])
    cfg["index"] = idx
    cfg.update(overrides)
    return cfg


def seed_for(idx: int) -> int:
    return BASE_SEED + idx


def bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns raw uint16 bits.

    Used only to store generated inputs (embedding tables, pre-filled caches)
    in the bf16 storage type the workload prescribes.
    """
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounding = 0x7FFF + ((u >> 16) & 1)
    out = ((u + rounding) >> 16).astype(np.uint16)
    nan = np.isnan(np.asarray(a, dtype=np.float32))
    if nan.any():
        out[nan] = 0x7FC0
    return out


def linear_shapes(cfg: dict) -> list[tuple[str, int, int]]:
    """(name, out, in) of every 4-bit linear, in generation order."""
    d, hd = cfg["dim"], cfg["head_dim"]
    qd, kd = cfg["n_heads"] * hd, cfg["n_kv_heads"] * hd
    f = cfg["ffn_dim"]
    out = []
    for l in range(cfg["n_layers"]):
        out += [(f"L{l}.wq", qd, d), (f"L{l}.wk", kd, d), (f"L{l}.wv", kd, d),
                (f"L{l}.wo", d, qd), (f"L{l}.w_gate", f, d), (f"L{l}.w_up", f, d),
                (f"L{l}.w_down", d, f)]
    if not cfg["tied"]:
        out.append(("lm_head", cfg["vocab"], d))
    return out


def _q4(rng: np.random.Generator, rows: int, cols: int) -> dict:
    assert cols % GROUP == 0
    # Each byte carries two independent uniform 0..15 codes.
    codes = rng.integers(0, 256, size=(rows, cols // 2), dtype=np.uint8)
    scale = rng.uniform(0.002, 0.006, size=(rows, cols // GROUP)).astype(np.float16)
    mins = (-7.5 * scale.astype(np.float64)).astype(np.float16)
    return dict(kind="q4", codes=codes, scales=scale, mins=mins, rows=rows, cols=cols)


def _norm(rng: np.random.Generator, n: int) -> dict:
    return dict(kind="f32", data=(1.0 + rng.normal(0.0, 0.01, size=n)).astype(np.float32),
                rows=1, cols=n)


def make_weights(cfg: dict, seed: int | None = None) -> dict:
    """All tensors of a workload, keyed by their canonical name."""
    if seed is None:
        seed = seed_for(cfg["index"])
    d, hd, V = cfg["dim"], cfg["head_dim"], cfg["vocab"]
    names = ["embed"]
    for l in range(cfg["n_layers"]):
        names += [f"L{l}.attn_norm", f"L{l}.wq", f"L{l}.wk", f"L{l}.wv"]
        if cfg["qk_norm"]:
            names += [f"L{l}.q_norm", f"L{l}.k_norm"]
        names += [f"L{l}.wo", f"L{l}.ffn_norm", f"L{l}.w_gate", f"L{l}.w_up", f"L{l}.w_down"]
    names.append("final_norm")
    if not cfg["tied"]:
        names.append("lm_head")
    children = np.random.SeedSequence(seed).spawn(len(names))
    shapes = {n: (o, i) for n, o, i in linear_shapes(cfg)}
    w = {}
    for name, ss in zip(names, children):
        rng = np.random.Generator(np.random.PCG64(ss))
        if name == "embed":
            e = rng.normal(0.0, 0.02, size=(V, d)).astype(np.float32)
            if cfg["tied"]:
                w[name] = dict(kind="bf16", data=bf16_bits_from_f32(e), rows=V, cols=d)
            else:
                w[name] = dict(kind="f32", data=e, rows=V, cols=d)
        elif name in shapes:
            w[name] = _q4(rng, *shapes[name])
        elif name.endswith("q_norm") or name.endswith("k_norm"):
            w[name] = _norm(rng, hd)
        else:
            w[name] = _norm(rng, d)
    return w


def make_prompt(cfg: dict, seed: int | None = None, n: int | None = None) -> np.ndarray:
    if seed is None:
        seed = seed_for(cfg["index"])
    n = cfg["prompt_len"] if n is None else n
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 1])))
    return rng.integers(0, cfg["vocab"], size=n, dtype=np.int32)


def make_first_tokens(cfg: dict, n_seq: int, seed: int | None = None) -> np.ndarray:
    """Seeded first decode token per sequence (workloads with a pre-filled cache)."""
    if seed is None:
        seed = seed_for(cfg["index"])
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 2])))
    return rng.integers(0, cfg["vocab"], size=n_seq, dtype=np.int32)


def make_kv_lengths(cfg: dict, n_seq: int, seed: int | None = None) -> np.ndarray:
    """Pre-filled cache length per sequence: fixed, or uniform in [lo, hi]."""
    if cfg.get("prefill_kv", 0) >= 0:
        return np.full(n_seq, cfg.get("prefill_kv", 0), dtype=np.int32)
    if seed is None:
        seed = seed_for(cfg["index"])
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 3])))
    return rng.integers(cfg["kv_len_lo"], cfg["kv_len_hi"] + 1, size=n_seq, dtype=np.int32)


def make_prefilled_kv(cfg: dict, layer: int, seq: int, n_pos: int,
                      seed: int | None = None) -> tuple[np.ndarray, np.ndarray]:
    """bf16 bits of N(0,1) keys and values, ``[n_pos][n_kv_heads][head_dim]`` each.

    Keys are taken as already rotated (the cache stores post-RoPE keys).
    """
    if seed is None:
        seed = seed_for(cfg["index"])
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 4, layer, seq])))
    shape = (n_pos, cfg["n_kv_heads"], cfg["head_dim"])
    k = bf16_bits_from_f32(rng.standard_normal(size=shape, dtype=np.float32))
    v = bf16_bits_from_f32(rng.standard_normal(size=shape, dtype=np.float32))
    return k, v


def weight_bytes(cfg: dict) -> dict:
    """Bytes of the per-token weight stream: 4-bit codes, fp16 scales+mins, bf16 LM head."""
    codes = scales = 0
    for _, o, i in linear_shapes(cfg):
        codes += o * i // 2
        scales += o * (i // GROUP) * 4
    lm16 = cfg["vocab"] * cfg["dim"] * 2 if cfg["tied"] else 0
    return dict(codes=codes, scales_mins=scales, lm_head_bf16=lm16, total=codes + scales + lm16)


def kv_bytes_per_pos(cfg: dict) -> int:
    """bf16 K+V bytes read per cached position per token (all layers)."""
    return 2 * cfg["n_layers"] * cfg["n_kv_heads"] * cfg["head_dim"] * 2
