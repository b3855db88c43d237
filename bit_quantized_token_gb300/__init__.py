"""Python binding of libllmq (the GB300 4-bit decode step).

Argument marshalling only: every step of the decode path runs in the CUDA
kernels of ``libllmq.so``. Loading fails loudly when the library is missing;
there is no CPU fallback. PyTorch is used by callers only for device memory
and streams (pass ``tensor.data_ptr()`` wherever a device pointer is
accepted).
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
# LLMQ_CHECKED=1 selects the checked build: every computed index into a weight
# stream, K/V cache row or partial-sum array is tested on the device, and one
# outside its buffer fails the call (LLM_ERR_CUDA, "an index left its buffer")
CHECKED = os.environ.get("LLMQ_CHECKED") == "1"
LIB_PATH = os.path.join(_HERE, "libllmq_checked.so" if CHECKED else "libllmq.so")
HEADER = os.path.join(_ROOT, "include", "llmq.h")
CSRC = os.path.join(_HERE, "csrc")


def sources() -> list[str]:
    """Every file the library is compiled from: the translation unit, all headers it may include, the ABI header."""
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh", ".h"))) + [HEADER]

ABI_VERSION = 1
LLM_F32, LLM_BF16, LLM_F16, LLM_Q4G64 = 0, 1, 2, 3
LLM_NO_GRAPH, LLM_NO_PDL, LLM_MULTI_KERNEL, LLM_DATAFLOW_STEP = 1, 2, 4, 8
LLM_DEBUG_BATCH_HIDDEN = 16
LLM_W4A8 = 64
LLM_KV_Q8 = 128
LLM_TEST_EXPIRE_WAIT = 0x80000000
STATUS = {0: "OK", -1: "INVALID_ARG", -2: "UNSUPPORTED", -3: "OOM", -4: "CTX_FULL", -5: "CUDA",
          -6: "TIMEOUT", -7: "NAN", -8: "NOT_FOUND"}

# Every entry point include/llmq.h declares.
EXPORTS = ["llm_model_create", "llm_model_destroy", "llm_prefill", "llm_prefill_batched", "llm_decode_step",
           "llm_decode_greedy", "llm_set_sampling",
           "llm_decode_step_batch", "llm_kv_reset", "llm_kv_write", "llm_kv_read", "llm_kv_read_q8", "llm_kv_len",
           "llm_debug_hidden", "llm_debug_unpack", "llm_model_stats", "llm_profile_step", "llm_time_kernel", "llm_sync",
           "llm_last_error", "llm_op_matvec", "llm_op_matvec_w4a8", "llm_matvec_noalloc", "llm_phase_times", "llm_debug_fail_alloc",
           "llm_debug_hidden_batch"]


# translation units of the library, compiled in parallel and linked into one shared object
UNITS = ["llmq.cu", "step_kernels.cu", "step_kernels_kv8.cu", "stepll_kernels.cu"]
BUILD_DIR = os.path.join(_HERE, "_build")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_compile_command(src: str, obj: str, defines=()) -> list[str]:
    return (["nvcc"] + ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-pthread",
                               "-I", os.path.join(_ROOT, "include")]
            + [f"-D{d}" for d in defines] + ["-c", "-o", obj, src])


def nvcc_link_command(objs: list[str], out: str) -> list[str]:
    return ["nvcc"] + ARCH + ["-shared", "-Xcompiler", "-fPIC,-pthread", "-o", out] + list(objs)


def build(force: bool = False, out: str | None = None, defines=()) -> str:
    """Compile libllmq.so in place for sm_103a (nvcc cross-compiles without a GPU).

    Rebuilds when the library is missing or older than any source; `out` and
    `defines` build a variant elsewhere (always rebuilt).
    """
    from concurrent.futures import ThreadPoolExecutor

    target = out or LIB_PATH
    if CHECKED and out is None:
        defines = list(defines) + ["LLMQ_CHECKED=1"]
    if out is None and not force and os.path.exists(LIB_PATH):
        newest = max(os.path.getmtime(f) for f in sources())
        if os.path.getmtime(LIB_PATH) >= newest:
            return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    tag = f"{os.getpid()}_{abs(hash(target)) % 100000}"
    objs = [os.path.join(BUILD_DIR, f"{u[:-3]}.{tag}.o") for u in UNITS]
    try:
        with ThreadPoolExecutor(len(UNITS)) as ex:
            futs = [ex.submit(subprocess.check_call, nvcc_compile_command(os.path.join(CSRC, u), o, defines))
                    for u, o in zip(UNITS, objs)]
            for f in futs:
                f.result()
        tmp = target + f".tmp{tag}"
        subprocess.check_call(nvcc_link_command(objs, tmp))
        os.replace(tmp, target)
    finally:
        for o in objs:
            if os.path.exists(o):
                os.unlink(o)
    return target


class LlmError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS.get(code, code)}: {msg}")
        self.code = code


class Config(C.Structure):
    _fields_ = [("abi_version", C.c_int32), ("dim", C.c_int32), ("n_layers", C.c_int32),
                ("n_heads", C.c_int32), ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32),
                ("ffn_dim", C.c_int32), ("vocab", C.c_int32), ("norm_eps", C.c_float),
                ("rope_neox", C.c_int32), ("rope_theta", C.c_double), ("qk_norm", C.c_int32),
                ("tied_embedding", C.c_int32), ("max_seq", C.c_int32), ("max_batch", C.c_int32),
                ("flags", C.c_uint32)]


class Tensor(C.Structure):
    _fields_ = [("name", C.c_char_p), ("dtype", C.c_int32), ("rows", C.c_int64), ("cols", C.c_int64),
                ("codes", C.c_void_p), ("scales", C.c_void_p), ("mins", C.c_void_p), ("data", C.c_void_p)]


class KernelTime(C.Structure):
    _fields_ = [("kind", C.c_int32), ("layer", C.c_int32), ("bytes", C.c_int64), ("ms", C.c_float)]


KERNEL_KINDS = {0: "gemv_q4", 1: "gemv_bf16", 2: "attention", 3: "argmax"}


class Stats(C.Structure):
    _fields_ = [("device_bytes", C.c_int64), ("weight_stream_bytes", C.c_int64),
                ("kv_bytes_per_pos", C.c_int64), ("kernels_per_step", C.c_int32), ("n_sm", C.c_int32)]


_lib = None


def lib() -> C.CDLL:
    """Load libllmq.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: run bit_quantized_token_gb300.build() (nvcc, sm_103a)")
        L = C.CDLL(LIB_PATH)
        P, i32 = C.c_void_p, C.c_int32
        sig = {
            "llm_model_create": (i32, [C.POINTER(Config), C.POINTER(Tensor), i32, P, C.POINTER(P)]),
            "llm_model_destroy": (None, [P]),
            "llm_prefill": (i32, [P, i32, P, i32, P, P]),
            "llm_prefill_batched": (i32, [P, i32, P, i32, P, P]),
            "llm_set_sampling": (i32, [P, C.c_float, i32, C.c_float, C.c_uint64]),
            "llm_decode_step": (i32, [P, i32, i32, P, P]),
            "llm_decode_greedy": (i32, [P, i32, i32, i32, P]),
            "llm_decode_step_batch": (i32, [P, P, i32, P, P]),
            "llm_kv_reset": (i32, [P, i32]),
            "llm_kv_write": (i32, [P, i32, i32, i32, i32, P, P]),
            "llm_kv_read": (i32, [P, i32, i32, i32, i32, P, P]),
            "llm_kv_read_q8": (i32, [P, i32, i32, i32, i32, P, P, P, P]),
            "llm_kv_len": (i32, [P, i32]),
            "llm_debug_hidden": (i32, [P, P]),
            "llm_debug_unpack": (i32, [P, C.c_char_p, P, P, P]),
            "llm_model_stats": (i32, [P, C.POINTER(Stats)]),
            "llm_profile_step": (i32, [P, i32, i32, C.POINTER(KernelTime), i32]),
            "llm_time_kernel": (i32, [P, i32, i32, i32, i32, C.POINTER(C.c_float), C.POINTER(C.c_int64)]),
            "llm_sync": (i32, [P]),
            "llm_last_error": (C.c_char_p, [P]),
            "llm_op_matvec": (i32, [C.POINTER(Tensor), P, P]),
            "llm_op_matvec_w4a8": (i32, [C.POINTER(Tensor), P, P]),
            "llm_matvec_noalloc": (i32, [P, C.c_char_p, P, P, P]),
            "llm_phase_times": (i32, [P, i32, i32, i32, P, C.c_int64]),
            "llm_debug_fail_alloc": (i32, [i32]),
            "llm_debug_hidden_batch": (i32, [P, P]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(rc: int, handle=None) -> None:
    if rc != 0:
        raise LlmError(rc, lib().llm_last_error(handle).decode())


def _ptr(a) -> int | None:
    """Raw address of a numpy array, a torch tensor or an int; None passes through."""
    if a is None:
        return None
    if isinstance(a, int):
        return a
    if isinstance(a, np.ndarray):
        assert a.flags["C_CONTIGUOUS"]
        return a.ctypes.data
    return a.data_ptr()  # torch tensor (host or device)


def tensor_table(weights: dict) -> tuple[C.Array, list]:
    """llm_tensor array for a dict name -> canonical tensor (see synth)."""
    keep = []
    arr = (Tensor * len(weights))()
    for i, (name, t) in enumerate(weights.items()):
        nm = name.encode()
        keep.append(nm)
        if t["kind"] == "q4":
            codes = np.ascontiguousarray(t["codes"], np.uint8)
            scales = np.ascontiguousarray(t["scales"]).view(np.uint16)
            mins = np.ascontiguousarray(t["mins"]).view(np.uint16)
            keep += [codes, scales, mins]
            arr[i] = Tensor(nm, LLM_Q4G64, t["rows"], t["cols"], codes.ctypes.data, scales.ctypes.data,
                            mins.ctypes.data, None)
        else:
            dt = LLM_BF16 if t["kind"] == "bf16" else LLM_F32
            data = np.ascontiguousarray(t["data"], np.uint16 if dt == LLM_BF16 else np.float32)
            keep.append(data)
            arr[i] = Tensor(nm, dt, t["rows"], t["cols"], None, None, None, data.ctypes.data)
    return arr, keep


def make_config(cfg: dict, max_seq: int, max_batch: int = 1, flags: int = 0) -> Config:
    return Config(ABI_VERSION, cfg["dim"], cfg["n_layers"], cfg["n_heads"], cfg["n_kv_heads"],
                  cfg["head_dim"], cfg["ffn_dim"], cfg["vocab"], float(cfg["norm_eps"]),
                  int(cfg["rope_neox"]), float(cfg["rope_theta"]), int(cfg["qk_norm"]),
                  int(cfg["tied"]), int(max_seq), int(max_batch), int(flags))


class Model:
    """Owner of one llm_model handle."""

    def __init__(self, cfg: dict, weights: dict, max_seq: int, max_batch: int = 1, flags: int = 0,
                 stream: int | None = None):
        self.cfg = cfg
        self.max_seq, self.max_batch = max_seq, max_batch
        conf = make_config(cfg, max_seq, max_batch, flags)
        table, keep = tensor_table(weights)
        h = C.c_void_p()
        rc = lib().llm_model_create(C.byref(conf), table, len(weights), stream, C.byref(h))
        del keep
        if rc != 0:
            raise LlmError(rc, lib().llm_last_error(None).decode())
        self.h = h

    def close(self) -> None:
        if getattr(self, "h", None):
            lib().llm_model_destroy(self.h)
            self.h = None

    def __del__(self):
        self.close()

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    # ---- decode ------------------------------------------------------------
    def prefill(self, seq: int, tokens, logits=None, argmax=None) -> None:
        toks = np.ascontiguousarray(tokens, np.int32)
        _check(lib().llm_prefill(self.h, seq, toks.ctypes.data, toks.size, _ptr(logits), _ptr(argmax)), self.h)

    def prefill_batched(self, seq: int, tokens, logits=None, argmax=None) -> None:
        """llm_prefill's contract, processed in chunks of up to 32 tokens."""
        toks = np.ascontiguousarray(tokens, np.int32)
        _check(lib().llm_prefill_batched(self.h, seq, toks.ctypes.data, toks.size, _ptr(logits), _ptr(argmax)),
               self.h)

    def set_sampling(self, temperature: float, top_k: int = 40, top_p: float = 0.95, seed: int = 42) -> None:
        """Sampled next-token choice for the batch-1 calls; temperature 0 = greedy."""
        _check(lib().llm_set_sampling(self.h, float(temperature), int(top_k), float(top_p), int(seed)), self.h)

    def decode_step(self, seq: int, token: int, logits=None, argmax=None) -> None:
        _check(lib().llm_decode_step(self.h, seq, int(token), _ptr(logits), _ptr(argmax)), self.h)

    def decode_greedy(self, seq: int, first_token: int, n_steps: int, tokens_out=None):
        out = np.empty(n_steps, np.int32) if tokens_out is None else tokens_out
        _check(lib().llm_decode_greedy(self.h, seq, int(first_token), int(n_steps), _ptr(out)), self.h)
        return out

    def decode_step_batch(self, tokens=None, logits=None, argmax=None) -> None:
        """One step of every sequence; tokens None = continue from the device-side greedy tokens."""
        if isinstance(tokens, (list, tuple)):
            tokens = np.ascontiguousarray(tokens, np.int32)
        _check(lib().llm_decode_step_batch(self.h, _ptr(tokens), self.max_batch, _ptr(logits), _ptr(argmax)),
               self.h)

    # ---- cache -------------------------------------------------------------
    def kv_reset(self, seq: int = -1) -> None:
        _check(lib().llm_kv_reset(self.h, seq), self.h)

    def kv_write(self, seq: int, layer: int, pos0: int, k_bits, v_bits) -> None:
        n = int(k_bits.shape[0])
        _check(lib().llm_kv_write(self.h, seq, layer, pos0, n, _ptr(k_bits), _ptr(v_bits)), self.h)

    def kv_read(self, seq: int, layer: int, pos0: int, n: int):
        shape = (n, self.cfg["n_kv_heads"], self.cfg["head_dim"])
        k = np.empty(shape, np.uint16)
        v = np.empty(shape, np.uint16)
        _check(lib().llm_kv_read(self.h, seq, layer, pos0, n, k.ctypes.data, v.ctypes.data), self.h)
        return k, v

    def kv_read_q8(self, seq: int, layer: int, pos0: int, n: int):
        """Codes [n, Hkv, hd] (int8) and fp16 scale bits [n, Hkv, hd/32] of K and V (int8 caches)."""
        H, hd = self.cfg["n_kv_heads"], self.cfg["head_dim"]
        k, v = np.empty((n, H, hd), np.int8), np.empty((n, H, hd), np.int8)
        ks, vs = np.empty((n, H, hd // 32), np.uint16), np.empty((n, H, hd // 32), np.uint16)
        _check(lib().llm_kv_read_q8(self.h, seq, layer, pos0, n, k.ctypes.data, ks.ctypes.data, v.ctypes.data,
                                    vs.ctypes.data), self.h)
        return k, ks, v, vs

    def kv_len(self, seq: int) -> int:
        r = lib().llm_kv_len(self.h, seq)
        if r < 0:
            raise LlmError(r, "kv_len")
        return r

    # ---- debug / info ------------------------------------------------------
    def hidden(self) -> np.ndarray:
        out = np.empty((self.cfg["n_layers"] + 1, self.cfg["dim"]), np.float32)
        _check(lib().llm_debug_hidden(self.h, out.ctypes.data), self.h)
        return out

    def hidden_batch(self) -> np.ndarray:
        """Per-layer residuals of the last batched step: [n_layers+1, max_batch, dim]."""
        out = np.empty((self.cfg["n_layers"] + 1, self.max_batch, self.cfg["dim"]), np.float32)
        _check(lib().llm_debug_hidden_batch(self.h, out.ctypes.data), self.h)
        return out

    def unpack(self, name: str, rows: int, cols: int):
        codes = np.empty((rows, cols // 2), np.uint8)
        scales = np.empty((rows, cols // 64), np.uint16)
        mins = np.empty((rows, cols // 64), np.uint16)
        _check(lib().llm_debug_unpack(self.h, name.encode(), codes.ctypes.data, scales.ctypes.data,
                                      mins.ctypes.data), self.h)
        return codes, scales, mins

    def stats(self) -> dict:
        s = Stats()
        _check(lib().llm_model_stats(self.h, C.byref(s)), self.h)
        return {f: getattr(s, f) for f, _ in Stats._fields_}

    def profile_step(self, seq: int, token: int) -> list[dict]:
        """One eager step with a CUDA-event pair around each kernel."""
        buf = (KernelTime * 4096)()
        n = lib().llm_profile_step(self.h, seq, int(token), buf, 4096)
        if n < 0:
            _check(n, self.h)
        return [dict(kind=KERNEL_KINDS[buf[i].kind], layer=buf[i].layer, bytes=buf[i].bytes, ms=buf[i].ms)
                for i in range(n)]

    KERNELS = {"qkv": 0, "attention": 1, "wo": 2, "gate_up": 3, "down": 4, "lm_head": 5, "all_gemv": 6}

    def time_kernel(self, seq: int, which: str, layer: int, n: int) -> tuple[float, int]:
        """Mean ms per launch of n back-to-back launches, and the launch's algorithmic bytes."""
        ms, nb = C.c_float(), C.c_int64()
        _check(lib().llm_time_kernel(self.h, seq, self.KERNELS[which], layer, n, C.byref(ms), C.byref(nb)),
               self.h)
        return float(ms.value), int(nb.value)

    def phase_times(self, seq: int, token: int, n_steps: int) -> np.ndarray:
        """Device timestamps (ns) of n_steps greedy steps through the flag-synchronised
        step: [n_steps][phases][n_sm][16]: SM cycles (clock64) when the input build starts, its inputs
        have arrived, the build is done, the units are done and the outputs are published; the largest
        per-warp cycles waiting for units and in unit dots, and their sums over the warps. Record
        [0][0][cta][12:16] holds (%globaltimer ns, clock64) at the kernel's start and end for the CTA."""
        n_sm = self.stats()["n_sm"]
        cap = 8 * 16 * 4096 * n_sm
        buf = np.zeros(cap, np.uint64)
        n = lib().llm_phase_times(self.h, seq, int(token), int(n_steps), buf.ctypes.data, cap)
        if n < 0:
            _check(n, self.h)
        return buf[:16 * n].reshape(n_steps, -1, n_sm, 16)

    def sync(self) -> None:
        _check(lib().llm_sync(self.h), self.h)


def matvec(t: dict, x) -> np.ndarray:
    """y = W x through the repack + dequant-GEMV kernel (W: canonical q4 or bf16 dict)."""
    table, keep = tensor_table({"w": t})
    x = np.ascontiguousarray(x, np.float32)
    y = np.empty(int(t["rows"]), np.float32)
    _check(lib().llm_op_matvec(table, x.ctypes.data, y.ctypes.data))
    return y


def matvec_w4a8(t: dict, x) -> np.ndarray:
    """y = W x in the W4A8 numerics (x quantized per 32-block to int8) through the GEMV kernel."""
    table, keep = tensor_table({"w": t})
    x = np.ascontiguousarray(x, np.float32)
    y = np.empty(int(t["rows"]), np.float32)
    _check(lib().llm_op_matvec_w4a8(table, x.ctypes.data, y.ctypes.data))
    return y


def debug_fail_alloc(nth: int) -> None:
    """Test hook: the nth device allocation of the models created next fails (0 disarms)."""
    _check(lib().llm_debug_fail_alloc(int(nth)))


def matvec_noalloc(model: Model, name: str, x, y, stream: int | None = None) -> None:
    """y = W x with a weight matrix resident in `model`; x, y are device buffers.

    Allocates no device memory (scratch is a static device array inside the
    library); see llm_matvec_noalloc in include/llmq.h.
    """
    _check(lib().llm_matvec_noalloc(model.h, name.encode(), _ptr(x), _ptr(y), stream), model.h)
