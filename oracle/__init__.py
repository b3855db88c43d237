"""CPU oracle for the 4-bit decode step -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library never loads it and
shares no code with it. The C source (``oracle.c``) is a plain fp64
restatement of the decoder the pages describe; this module is ctypes glue that
hands it numpy arrays in the canonical packed layout.

Parity pins: tests/test_oracle_pins.py checks every exported function against
closed forms, brute force on tiny inputs, golden fixtures and the
prefix-versus-cache invariant, and checks that planted mistakes are caught.
"""
from __future__ import annotations

import contextlib
import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

MUT = dict(none=0, rope_pairing=1, mask_polarity=2, cache_frontier=3, qk_orientation=4,
           gqa_map=5, nibble_order=6, scale_min_swap=7, no_residual=8, rope_sign=9)


def build(force: bool = False) -> str:
    """Compile liboracle.so in place (gcc, OpenMP, strict IEEE: no fp contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < max(
            os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "oracle.h"))):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=gnu11", "-ffp-contract=off", "-fno-fast-math",
                               "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib() -> C.CDLL:
    global _lib
    if _lib is None:
        build()
        _lib = C.CDLL(_LIB)
        _declare(_lib)
    return _lib


class Q4(C.Structure):
    _fields_ = [("codes", C.c_void_p), ("scales", C.c_void_p), ("mins", C.c_void_p),
                ("rows", C.c_int64), ("cols", C.c_int64)]


class Config(C.Structure):
    _fields_ = [("dim", C.c_int32), ("n_layers", C.c_int32), ("n_heads", C.c_int32),
                ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32), ("ffn_dim", C.c_int32),
                ("vocab", C.c_int32), ("rope_neox", C.c_int32), ("qk_norm", C.c_int32),
                ("tied", C.c_int32), ("embed_bf16", C.c_int32), ("pad_", C.c_int32),
                ("norm_eps", C.c_double), ("rope_theta", C.c_double)]


class Layer(C.Structure):
    _fields_ = [("wq", Q4), ("wk", Q4), ("wv", Q4), ("wo", Q4), ("wg", Q4), ("wu", Q4),
                ("wd", Q4), ("attn_norm", C.c_void_p), ("ffn_norm", C.c_void_p),
                ("q_norm", C.c_void_p), ("k_norm", C.c_void_p)]


class Model(C.Structure):
    _fields_ = [("cfg", Config), ("embed", C.c_void_p), ("final_norm", C.c_void_p),
                ("lm_head", Q4), ("layers", C.POINTER(Layer))]


class Cache(C.Structure):
    _fields_ = [("k", C.c_void_p), ("v", C.c_void_p), ("cap", C.c_int32), ("len", C.c_int32),
                ("k8", C.c_void_p), ("v8", C.c_void_p), ("ks", C.c_void_p), ("vs", C.c_void_p)]


Q8_GROUP = 32


def _declare(L: C.CDLL) -> None:
    P, i32, i64, d = C.c_void_p, C.c_int32, C.c_int64, C.c_double
    sig = {
        "orc_set_mutation": (None, [i32]),
        "orc_num_threads": (i32, []),
        "orc_half_to_double": (d, [C.c_uint16]),
        "orc_bf16_to_double": (d, [C.c_uint16]),
        "orc_bf16_from_double": (C.c_uint16, [d]),
        "orc_f32_from_double": (C.c_float, [d]),
        "orc_dequant_row": (None, [P, i64, P]),
        "orc_matvec": (None, [P, P, P]),
        "orc_rmsnorm": (None, [P, P, i32, d, P]),
        "orc_rope": (None, [P, i32, i32, d, i32]),
        "orc_silu_mul": (None, [P, P, i32, P]),
        "orc_attend": (None, [P, P, P, i32, i32, P]),
        "orc_half_from_float": (C.c_uint16, [C.c_float]),
        "orc_q8_quantize": (None, [P, i32, P, P]),
        "orc_q8_value": (d, [C.c_int8, C.c_uint16]),
        "orc_attend_q8": (None, [P, P, P, P, P, i32, i32, P]),
        "orc_set_kv_q8": (None, [i32]),
        "orc_argmax_f32": (i32, [P, i64]),
        "orc_step": (i32, [P, P, i32, P, P]),
        "orc_full_prefix": (i32, [P, P, i32, P, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float64)


def num_threads() -> int:
    return int(lib().orc_num_threads())


def set_mutation(m: int | str) -> None:
    lib().orc_set_mutation(MUT[m] if isinstance(m, str) else int(m))


@contextlib.contextmanager
def mutation(m: int | str):
    """Plant one of the oracle's mistakes for the duration of a block (tests only)."""
    set_mutation(m)
    try:
        yield
    finally:
        set_mutation(0)


def half_to_double(bits: int) -> float:
    return float(lib().orc_half_to_double(int(bits)))


def half_from_float(x: float) -> int:
    return int(lib().orc_half_from_float(float(x)))


def q8_quantize(x) -> tuple[np.ndarray, np.ndarray]:
    """Grouped int8 codes [n] and fp16 scale bits [n / 32] of a vector (n a multiple of 32)."""
    x = _f64(x)
    assert x.size % Q8_GROUP == 0
    q = np.empty(x.size, dtype=np.int8)
    dd = np.empty(x.size // Q8_GROUP, dtype=np.uint16)
    lib().orc_q8_quantize(_ptr(x), x.size, _ptr(q), _ptr(dd))
    return q, dd


def q8_values(q: np.ndarray, d: np.ndarray) -> np.ndarray:
    """Stored values of grouped int8 codes: code x fp16 scale, exactly."""
    return np.array([lib().orc_q8_value(int(c), int(d[i // Q8_GROUP])) for i, c in enumerate(q)])


def attend_q8(q, k8, ks, v8, vs) -> np.ndarray:
    """orc_attend over grouped-int8 rows: k8/v8 [n_pos][hd] int8, ks/vs [n_pos][hd/32] fp16 bits."""
    q = _f64(q)
    k8, v8 = (np.ascontiguousarray(a, dtype=np.int8) for a in (k8, v8))
    ks, vs = (np.ascontiguousarray(a, dtype=np.uint16) for a in (ks, vs))
    out = np.empty(q.size, dtype=np.float64)
    lib().orc_attend_q8(_ptr(q), _ptr(k8), _ptr(ks), _ptr(v8), _ptr(vs), k8.shape[0], q.size, _ptr(out))
    return out


@contextlib.contextmanager
def kv_q8():
    """Full-prefix mode with grouped int8 K/V for the duration of a block."""
    lib().orc_set_kv_q8(1)
    try:
        yield
    finally:
        lib().orc_set_kv_q8(0)


def bf16_to_double(bits: int) -> float:
    return float(lib().orc_bf16_to_double(int(bits)))


def bf16_from_double(x: float) -> int:
    return int(lib().orc_bf16_from_double(float(x)))


def _q4(t: dict) -> tuple[Q4, list]:
    codes = np.ascontiguousarray(t["codes"], dtype=np.uint8)
    scales = np.ascontiguousarray(t["scales"]).view(np.uint16)
    mins = np.ascontiguousarray(t["mins"]).view(np.uint16)
    q = Q4(_ptr(codes), _ptr(scales), _ptr(mins), int(t["rows"]), int(t["cols"]))
    return q, [codes, scales, mins]


def dequant_row(t: dict, r: int) -> np.ndarray:
    q, keep = _q4(t)
    out = np.empty(int(t["cols"]), dtype=np.float64)
    lib().orc_dequant_row(C.byref(q), int(r), _ptr(out))
    return out


def matvec(t: dict, x) -> np.ndarray:
    q, keep = _q4(t)
    x = _f64(x)
    assert x.shape == (int(t["cols"]),)
    y = np.empty(int(t["rows"]), dtype=np.float64)
    lib().orc_matvec(C.byref(q), _ptr(x), _ptr(y))
    return y


def rmsnorm(x, w, eps: float) -> np.ndarray:
    x = _f64(x)
    w = np.ascontiguousarray(w, dtype=np.float32)
    out = np.empty_like(x)
    lib().orc_rmsnorm(_ptr(x), _ptr(w), x.size, float(eps), _ptr(out))
    return out


def rope(v, pos: int, theta: float, neox: int) -> np.ndarray:
    v = _f64(v).copy()
    lib().orc_rope(_ptr(v), v.size, int(pos), float(theta), int(neox))
    return v


def silu_mul(g, u) -> np.ndarray:
    g, u = _f64(g), _f64(u)
    out = np.empty_like(g)
    lib().orc_silu_mul(_ptr(g), _ptr(u), g.size, _ptr(out))
    return out


def attend(q, k_bits, v_bits) -> np.ndarray:
    """One query head over bf16 key/value rows ``[n_pos][hd]`` (raw uint16 bits)."""
    q = _f64(q)
    k = np.ascontiguousarray(k_bits, dtype=np.uint16)
    v = np.ascontiguousarray(v_bits, dtype=np.uint16)
    n_pos, hd = k.shape
    out = np.empty(hd, dtype=np.float64)
    lib().orc_attend(_ptr(q), _ptr(k), _ptr(v), n_pos, hd, _ptr(out))
    return out


def argmax_f32(logits) -> int:
    lg = _f64(logits)
    return int(lib().orc_argmax_f32(_ptr(lg), lg.size))


class OracleModel:
    """fp64 decoder over canonical weights (dict name -> tensor dict, see synth)."""

    def __init__(self, cfg: dict, weights: dict):
        self.cfg = cfg
        self._keep = []
        L = cfg["n_layers"]
        layers = (Layer * L)()
        for l in range(L):
            lay = layers[l]
            for fld, nm in (("wq", "wq"), ("wk", "wk"), ("wv", "wv"), ("wo", "wo"),
                            ("wg", "w_gate"), ("wu", "w_up"), ("wd", "w_down")):
                q, keep = _q4(weights[f"L{l}.{nm}"])
                setattr(lay, fld, q)
                self._keep += keep
            for fld in ("attn_norm", "ffn_norm", "q_norm", "k_norm"):
                key = f"L{l}.{fld}"
                if key in weights:
                    a = np.ascontiguousarray(weights[key]["data"], dtype=np.float32)
                    self._keep.append(a)
                    setattr(lay, fld, _ptr(a))
        self._layers = layers
        emb = weights["embed"]
        embed_bf16 = 1 if emb["kind"] == "bf16" else 0
        e = np.ascontiguousarray(emb["data"], dtype=np.uint16 if embed_bf16 else np.float32)
        fn = np.ascontiguousarray(weights["final_norm"]["data"], dtype=np.float32)
        self._keep += [e, fn]
        lm = Q4()
        if not cfg["tied"]:
            lm, keep = _q4(weights["lm_head"])
            self._keep += keep
        conf = Config(cfg["dim"], L, cfg["n_heads"], cfg["n_kv_heads"], cfg["head_dim"],
                      cfg["ffn_dim"], cfg["vocab"], cfg["rope_neox"], cfg["qk_norm"],
                      cfg["tied"], embed_bf16, 0, float(cfg["norm_eps"]), float(cfg["rope_theta"]))
        self._model = Model(conf, _ptr(e), _ptr(fn), lm, layers)

    def new_cache(self, cap: int, kv: str = "bf16") -> "OracleCache":
        return OracleCache(self.cfg, cap, kv)

    def step(self, cache: "OracleCache", tok: int, hidden: bool = False):
        cfg = self.cfg
        logits = np.empty(cfg["vocab"], dtype=np.float64)
        hid = np.empty((cfg["n_layers"] + 1, cfg["dim"]), dtype=np.float64) if hidden else None
        rc = lib().orc_step(C.byref(self._model), C.byref(cache.c), int(tok), _ptr(logits),
                            _ptr(hid) if hidden else None)
        if rc != 0:
            raise ValueError(f"oracle step failed (pos={cache.c.len}, cap={cache.c.cap}, tok={tok})")
        return (logits, hid) if hidden else logits

    def full_prefix(self, toks, hidden: bool = False):
        cfg = self.cfg
        toks = np.ascontiguousarray(toks, dtype=np.int32)
        n = toks.size
        logits = np.empty((n, cfg["vocab"]), dtype=np.float64)
        hid = np.empty((cfg["n_layers"] + 1, n, cfg["dim"]), dtype=np.float64) if hidden else None
        rc = lib().orc_full_prefix(C.byref(self._model), _ptr(toks), n, _ptr(logits),
                                   _ptr(hid) if hidden else None)
        if rc != 0:
            raise ValueError("oracle full-prefix failed")
        return (logits, hid) if hidden else logits


class OracleCache:
    """K/V storage of one sequence: ``[n_layers][n_kv_heads][cap][head_dim]`` bf16,
    or (kv="q8") int8 codes with fp16 scales ``[...][head_dim / 32]``."""

    def __init__(self, cfg: dict, cap: int, kv: str = "bf16"):
        shape = (cfg["n_layers"], cfg["n_kv_heads"], cap, cfg["head_dim"])
        self.k = np.zeros(shape, dtype=np.uint16)
        self.v = np.zeros(shape, dtype=np.uint16)
        self.c = Cache(_ptr(self.k), _ptr(self.v), cap, 0)
        if kv == "q8":
            self.k8 = np.zeros(shape, dtype=np.int8)
            self.v8 = np.zeros(shape, dtype=np.int8)
            sshape = shape[:3] + (cfg["head_dim"] // Q8_GROUP,)
            self.ks = np.zeros(sshape, dtype=np.uint16)
            self.vs = np.zeros(sshape, dtype=np.uint16)
            self.c.k8, self.c.v8 = _ptr(self.k8), _ptr(self.v8)
            self.c.ks, self.c.vs = _ptr(self.ks), _ptr(self.vs)
        else:
            assert kv == "bf16", kv

    @property
    def len(self) -> int:
        return int(self.c.len)

    def fill(self, layer: int, k_bits: np.ndarray, v_bits: np.ndarray, pos0: int = 0) -> None:
        """Write bf16 rows ``[n][n_kv_heads][hd]`` at positions pos0.. of one layer.

        An int8 cache stores each (position, head) row through the grouped
        int8 quantizer (q8_quantize) of its bf16 values.
        """
        n = k_bits.shape[0]
        self.k[layer, :, pos0:pos0 + n, :] = np.transpose(k_bits, (1, 0, 2))
        self.v[layer, :, pos0:pos0 + n, :] = np.transpose(v_bits, (1, 0, 2))
        if hasattr(self, "k8"):
            for bits, codes, scales in ((k_bits, self.k8, self.ks), (v_bits, self.v8, self.vs)):
                vals = (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
                rows = np.ascontiguousarray(np.transpose(vals, (1, 0, 2)))  # [head][position][hd]
                c, d = q8_quantize(rows.reshape(-1))  # groups of 32 never straddle a row (hd % 32 == 0)
                H, hd = rows.shape[0], rows.shape[2]
                codes[layer, :, pos0:pos0 + n, :] = c.reshape(H, n, hd)
                scales[layer, :, pos0:pos0 + n, :] = d.reshape(H, n, hd // Q8_GROUP)

    def set_len(self, n: int) -> None:
        self.c.len = int(n)


def greedy_run(model: OracleModel, prompt, n_steps: int, cap: int | None = None,
               hidden: bool = False, kv: str = "bf16"):
    """prefill(prompt) -> t0 = argmax, then n_steps cached steps feeding back argmax.

    Returns tokens [n_steps+1], logits [n_steps+1][vocab] and, if asked, the
    hidden states of every step. kv: the cache's storage ("bf16" or "q8").
    """
    prompt = list(int(t) for t in prompt)
    cap = cap or (len(prompt) + n_steps + 1)
    cache = model.new_cache(cap, kv)
    hids = []
    for t in prompt[:-1]:
        model.step(cache, t)
    toks, logs = [], []
    cur = prompt[-1]
    for i in range(n_steps + 1):
        r = model.step(cache, cur, hidden=hidden)
        lg, hd = (r if hidden else (r, None))
        nxt = argmax_f32(lg)
        toks.append(nxt)
        logs.append(lg)
        if hidden:
            hids.append(hd)
        cur = nxt
    out = dict(tokens=np.array(toks, dtype=np.int32), logits=np.array(logs), cache=cache)
    if hidden:
        out["hidden"] = np.array(hids)
    return out
