"""Host-side checks of the C ABI: the library loads without a GPU, exports every
entry point include/llmq.h declares, and the ctypes structs match the C layout."""
import os
import re
import subprocess

import pytest

import bit_quantized_token_gb300 as bq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def library():
    bq.build()
    return bq.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "llmq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\**(llm_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_binding_surface():
    assert declared_functions() == sorted(bq.EXPORTS)


def test_library_exports_every_declared_symbol(library):
    for name in declared_functions():
        assert hasattr(library, name), name


def test_errors_without_gpu_work(library):
    # argument validation happens before any device call
    rc = library.llm_model_create(None, None, 0, None, None)
    assert rc == -1
    assert b"null" in library.llm_last_error(None)
    assert library.llm_kv_len(None, 0) == -1


def test_struct_layouts_match_c(tmp_path):
    prog = tmp_path / "layout.c"
    prog.write_text("""
#include <stddef.h>
#include <stdio.h>
#include "llmq.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu\\n", sizeof(llm_config), offsetof(llm_config, norm_eps),
         offsetof(llm_config, rope_theta), offsetof(llm_config, max_seq), offsetof(llm_config, flags));
  printf("%zu %zu %zu\\n", sizeof(llm_tensor), offsetof(llm_tensor, rows), offsetof(llm_tensor, data));
  printf("%zu %zu\\n", sizeof(llm_stats), offsetof(llm_stats, kernels_per_step));
  return 0;
}
""")
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-I", os.path.join(ROOT, "include"), str(prog), "-o", str(exe)])
    lines = subprocess.check_output([str(exe)]).decode().split("\n")
    C = bq.Config
    assert lines[0].split() == [str(x) for x in (C.__sizeof__(C()) if False else __import__("ctypes").sizeof(C),
                                                 C.norm_eps.offset, C.rope_theta.offset, C.max_seq.offset,
                                                 C.flags.offset)]
    T = bq.Tensor
    assert lines[1].split() == [str(x) for x in (__import__("ctypes").sizeof(T), T.rows.offset, T.data.offset)]
    S = bq.Stats
    assert lines[2].split() == [str(x) for x in (__import__("ctypes").sizeof(S), S.kernels_per_step.offset)]


def test_build_command_targets_sm103a():
    for u in bq.UNITS:
        cmd = " ".join(bq.nvcc_compile_command(u, "x.o"))
        assert "arch=compute_103a,code=sm_103a" in cmd and " -c " in cmd and "-O3" in cmd
    link = " ".join(bq.nvcc_link_command(["a.o", "b.o"], "x.so"))
    assert "arch=compute_103a,code=sm_103a" in link and "-shared" in link


def test_flags_statuses_and_dtypes_match_the_header():
    import re
    text = open(bq.HEADER).read()
    flags = {n: int(v, 0) for n, v in re.findall(r"^#define (LLM_[A-Z0-9_]+)\s+(0x[0-9a-fA-F]+|\d+)u", text, re.M)}
    assert flags, "no flags found"
    for name, value in flags.items():
        assert getattr(bq, name) == value, name
    statuses = {int(v): n for n, v in re.findall(r"(LLM_(?:OK|ERR_[A-Z_]+))\s*=\s*(-?\d+)", text)}
    assert {k: v.replace("LLM_ERR_", "").replace("LLM_", "") for k, v in statuses.items()} == bq.STATUS
    dtypes = dict(re.findall(r"(LLM_(?:F32|BF16|F16|Q4G64))\s*=\s*(\d+)", text))
    assert dtypes and all(getattr(bq, n) == int(v) for n, v in dtypes.items())
