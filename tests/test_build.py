"""build() recompiles the library whenever any file it is compiled from changes.

CPU only: the compiler call is replaced by a recorder that writes the output
file, and the sources are copies in a temporary tree, so nothing here runs
nvcc or touches the real tree's timestamps.
"""
import os
import re
import shutil

import bit_quantized_token_gb300 as bq


def _includes(path):
    with open(path) as f:
        return re.findall(r'^\s*#\s*include\s+"([^"]+)"', f.read(), re.M)


def test_sources_cover_every_local_include():
    names = {os.path.basename(p) for p in bq.sources()}
    todo = [os.path.join(bq.CSRC, "llmq.cu")]
    seen = set()
    while todo:
        p = todo.pop()
        if p in seen:
            continue
        seen.add(p)
        for inc in _includes(p):
            assert os.path.basename(inc) in names, f"{p} includes {inc}, which build() does not track"
            local = os.path.join(bq.CSRC, inc)
            todo.append(local if os.path.exists(local) else bq.HEADER)
    assert os.path.join(bq.CSRC, "llmq.cu") in bq.sources() and bq.HEADER in bq.sources()


def test_touching_any_source_rebuilds(tmp_path, monkeypatch):
    csrc = tmp_path / "csrc"
    shutil.copytree(bq.CSRC, csrc, ignore=shutil.ignore_patterns("*.so", "*.o"))
    inc = tmp_path / "include"
    inc.mkdir()
    shutil.copy(bq.HEADER, inc / "llmq.h")
    lib = tmp_path / "libllmq.so"
    monkeypatch.setattr(bq, "CSRC", str(csrc))
    monkeypatch.setattr(bq, "HEADER", str(inc / "llmq.h"))
    monkeypatch.setattr(bq, "LIB_PATH", str(lib))
    monkeypatch.setattr(bq, "BUILD_DIR", str(tmp_path / "_build"))
    calls = []  # one entry per library link (each preceded by a compile of every unit)
    compiled = []

    def fake_compile(cmd, *a, **k):
        out = cmd[cmd.index("-o") + 1]
        with open(out, "w") as f:
            f.write("built")
        if "-shared" in cmd:
            assert len(compiled) == len(bq.UNITS) and all(o in cmd for o in compiled)
            compiled.clear()
            calls.append(out)
        else:
            compiled.append(out)
        return 0

    monkeypatch.setattr(bq.subprocess, "check_call", fake_compile)
    srcs = bq.sources()
    assert len(srcs) >= 8 and all(p.startswith(str(tmp_path)) for p in srcs)
    t0 = 1_700_000_000
    for p in srcs:
        os.utime(p, (t0, t0))
    bq.build()  # no library yet
    assert len(calls) == 1 and lib.exists()
    os.utime(lib, (t0 + 10, t0 + 10))
    bq.build()  # up to date
    assert len(calls) == 1
    for i, p in enumerate(srcs):
        t = t0 + 20 + 10 * i
        os.utime(p, (t, t))  # this source edited after the library was built
        bq.build()
        assert len(calls) == 2 + i, f"editing {os.path.basename(p)} did not rebuild"
        os.utime(lib, (t + 5, t + 5))
    bq.build(force=True)
    assert len(calls) == 2 + len(srcs)
