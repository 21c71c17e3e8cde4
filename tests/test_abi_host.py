"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every symbol the header declares, and validates arguments before touching
CUDA.  Plus the separation rule: the product path never imports the oracle."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from skinny_gemm_q4_gb300 import build, qgemv
    build.build()
    return qgemv.load()


def _declared():
    with open(os.path.join(ROOT, "include", "qgemv.h")) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(qgemv_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    from skinny_gemm_q4_gb300 import qgemv
    names = _declared()
    assert len(names) >= 12
    assert sorted(names) == sorted(qgemv.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n


CITES = re.compile(r'"docs/kernels\.md"|"docs/performance\.md"|"Kernels"|no counterpart')


def test_every_declaration_cites_its_passage():
    """Each exported call's comment in include/qgemv.h names the page passage
    that defines it (or says that the pages have no counterpart)."""
    with open(os.path.join(ROOT, "include", "qgemv.h")) as f:
        src = f.read()
    found = 0
    for m in re.finditer(r"/\*((?:(?!\*/).)*)\*/\s*\n(?:[^;/]*?)\b(qgemv_[a-z_]+)\s*\(", src,
                         re.S):
        comment, name = m.group(1), m.group(2)
        assert CITES.search(comment), f"{name}: no citation in its comment"
        found += 1
    assert found == len(_declared())


def test_row_bytes_and_describe(lib):
    from skinny_gemm_q4_gb300 import qgemv as q
    assert q.qgemv_row_bytes(q.Q4_K, 2560) == 1440
    assert q.qgemv_row_bytes(q.Q5_K, 9728) == 6688
    assert q.qgemv_row_bytes(q.Q6_K, 9728) == 7980
    assert q.qgemv_row_bytes(q.NVFP4_W4A16, 27648) == 13824
    assert q.qgemv_row_bytes(q.Q4_K, 100) == -1
    assert q.qgemv_row_bytes(7, 256) == -1
    d = q.qgemv_describe()
    assert "Q4_K=12" in d and "QGEMV_FAULT_INJECT" in d


def _create(lib, t, M, K, w, sc=None, g=1.0, flags=0):
    from skinny_gemm_q4_gb300 import qgemv as q
    h = ctypes.c_void_p()
    opts = q.QgOpts(flags, 0)
    st = lib.qgemv_create(ctypes.byref(h), t, M, K, w, sc, g, ctypes.byref(opts))
    return st, h


def test_create_validates_before_cuda(lib, monkeypatch):
    from skinny_gemm_q4_gb300 import qgemv as q
    assert _create(lib, q.Q4_K, 16, 2560, None)[0] == -1          # null weights
    assert _create(lib, q.Q4_K, 16, 2500, 256)[0] == -2           # K % 256
    assert _create(lib, 99, 16, 2560, 256)[0] == -2               # unknown type
    assert _create(lib, q.Q4_K, 0, 2560, 256)[0] == -1            # M
    assert _create(lib, q.Q4_K, 16, 2560, 258)[0] == -3           # alignment
    assert _create(lib, q.NVFP4_W4A16, 16, 2560, 256, None)[0] == -1
    assert _create(lib, q.NVFP4_W4A16, 16, 2560, 256, 264)[0] == -3
    assert _create(lib, q.NVFP4_W4A16, 16, 2560, 256, 512, float("nan"))[0] == -1
    assert "finite" in q.qgemv_last_error()
    monkeypatch.setenv("QGEMV_FAULT_INJECT", "create")
    assert _create(lib, q.Q4_K, 16, 2560, 256)[0] == -6
    assert "injected" in q.qgemv_last_error()


def test_null_handle_calls_are_errors(lib):
    assert lib.qgemv_run(None, 16, 1, 16, 0, None) == -1
    assert lib.qgemv_dequantize(None, 16, None) == -1
    assert lib.qgemv_run_host(None, 16, 1, 16, 0, None) == -1
    lib.qgemv_destroy(None)
    from skinny_gemm_q4_gb300 import qgemv as q
    calls = q.make_calls([(q.CALL_RUN, [None], 16, 1, [16], 0, None)])
    assert lib.qgemv_chain_run(None, calls, 1, None) == -1
    assert lib.qgemv_chain_status(None, None, 0) == -1
    assert lib.qgemv_chain_run_host(None, calls, 1, None, None, 0, None, None, 0, None) == -1
    lib.qgemv_chain_destroy(None)


def test_product_path_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "skinny_gemm_q4_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".c")):
                with open(os.path.join(dirpath, f)) as fh:
                    src = fh.read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", src, re.M), f
                assert "oracle.h" not in src and "oracle/" not in src, f


def test_generators_are_seeded_and_shaped():
    from skinny_gemm_q4_gb300 import synth
    a = synth.q4k_weights(8, 512, seed=1, stream=2)
    b = synth.q4k_weights(8, 512, seed=1, stream=2)
    c = synth.q4k_weights(8, 512, seed=1, stream=3)
    assert a.shape == (8, 288) and np.array_equal(a, b) and not np.array_equal(a, c)
    q6 = synth.q6k_weights(4, 256, seed=0)
    sc = q6[:, 192:208].view(np.int8)
    assert q6.shape == (4, 210) and sc.min() >= -128 and sc.max() <= 127
    d = q6[:, 208:210].copy().view(np.float16)
    assert np.all(d >= 0)
    codes, scales, g = synth.nvfp4_weights(4, 512, seed=0)
    assert codes.shape == (4, 256) and scales.shape == (4, 32) and 0.5 <= g < 1.0
    assert scales.min() >= 0x08 and scales.max() <= 0x58
    x = synth.activations(9, 64, seed=0, duplicate_rows=True)
    assert np.array_equal(x[2], x[0]) and np.array_equal(x[5], x[3]) and np.array_equal(x[8], x[6])


_NOALLOC_PROBE = r"""
import ctypes, sys
sys.path.insert(0, sys.argv[1])
from skinny_gemm_q4_gb300 import qgemv as q
lib = q.load()
f = lib.qgemv_run_noalloc
def call(t, M, K, w, sc, g, x, N, y, ydt=0):
    st = f(t, M, K, w, sc, g, x, N, y, ydt, None)
    return st, q.qgemv_last_error()
out = []
out.append(call(q.Q4_K, 16, 1 << 20, 4096, None, 1.0, 4096, 1, 4096))          # K > 931,840
out.append(call(q.NVFP4_W4A16, 16, 2560, 4096, 8192, float("nan"), 4096, 1, 4096))
out.append(call(q.Q4_K, 64 * 65536, 2560, 4096, None, 1.0, 4096, 1, 4096))     # grid rows
out.append(call(q.Q4_K, 16, 2560, 4100, None, 1.0, 4096, 1, 4096))            # w alignment
out.append(call(q.Q4_K, 16, 2560, 4096, None, 1.0, 4100, 1, 4096))            # x alignment
out.append(call(q.Q4_K, 16, 2560, 4096, None, 1.0, 4096, 0, 4096))            # N
out.append(call(q.Q4_K, 16, 2560, None, None, 1.0, 4096, 1, 4096))            # null w
out.append(call(77, 16, 2560, 4096, None, 1.0, 4096, 1, 4096))                 # type
out.append(call(q.Q4_K, 16, 2500, 4096, None, 1.0, 4096, 1, 4096))            # K % 256
for st, msg in out:
    print(st, "|", msg)
"""


def test_noalloc_validates_before_touching_the_device(lib, tmp_path):
    """Every argument check of qgemv_run_noalloc runs before any CUDA call:
    with no visible device (and fake addresses) each bad call returns its
    validation status, never a CUDA error and never a launch."""
    import subprocess
    import sys
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", _NOALLOC_PROBE, ROOT], env=env,
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    rows = [line.split(" | ", 1) for line in r.stdout.strip().splitlines()]
    st = [int(a) for a, _ in rows]
    msg = [b for _, b in rows]
    assert st == [-2, -1, -2, -3, -3, -1, -1, -2, -2], rows
    assert "2097152-byte" in msg[0] or "scratch" in msg[0]
    assert "finite" in msg[1]
    assert "rows" in msg[2]
