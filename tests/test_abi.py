"""The C-ABI library builds, loads and exports what include/pagedattn.h declares;
its host-side argument checks reject bad calls before touching the GPU.

Nothing here launches a kernel, so it runs without a GPU.
"""
import ctypes
import glob
import os
import re

import pytest

import paged_kv_cache_305_gb300 as pa
from paged_kv_cache_305_gb300 import build as pbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names.update(re.findall(r"\b(pa_\w+)\s*\(", text))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    pbuild.build()
    return pa.load_library()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert {"pa_decode", "pa_reshape_and_cache", "pa_decode_workspace_bytes", "pa_last_error"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
    assert set(pa.pagedattn.EXPORTED) <= set(names)


def test_header_compiles_and_links_as_plain_c(lib, tmp_path):
    # the boundary is a C ABI: the header compiles as C99 (no C++), and a C
    # program links against the library and gets the same host-side answer
    # as the Python binding (workspace sizing needs no GPU)
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    cuda_inc = None
    for d in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        if d and os.path.exists(os.path.join(d, "include", "cuda_runtime_api.h")):
            cuda_inc = os.path.join(d, "include")
            break
    if gcc is None or cuda_inc is None:
        pytest.skip("gcc or the CUDA headers are not available")
    libdir = os.path.dirname(pbuild.LIB_PATH)
    src = tmp_path / "use_header.c"
    src.write_text('#include "pagedattn.h"\n#include <stdio.h>\n'
                   "int main(void) {\n"
                   "  printf(\"%zu\\n\", pa_decode_workspace_bytes(4, 8, 128, 64, 16, 512));\n"
                   "  return pa_last_error() == 0;\n"
                   "}\n")
    exe = tmp_path / "use_header"
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                        "-I", cuda_inc, str(src), "-L", libdir, "-lpagedattn",
                        "-Wl,-rpath," + libdir, "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    assert int(out.stdout.strip()) == pa.decode_workspace_bytes(4, 8, 128, 64, 16, 512)


def test_library_is_built_for_sm_103a_only():
    assert pbuild.ARCH_FLAGS == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_workspace_bytes_arithmetic(lib):
    # a 256-byte header (claim counter, finished CTAs), S * Hq counters, then
    # S * Hq * P lse values, then S * Hq * P * d outputs (fp32)
    def expect(S, Hq, d, MB, B, pt):
        # partition_tokens 0: 1024 when the table addresses 4096+ tokens, else 512
        default = 1024 if MB * B >= 4096 else 512
        P = -(-(MB * B) // (pt or default))
        if P <= 1:
            return 0
        r = lambda x: -(-x // 256) * 256
        rows = S * Hq
        return r(256 + rows * 4) + r(rows * P * 4) + rows * P * d * 4
    for args in [(128, 32, 128, 512, 16, 0), (8, 64, 128, 8192, 16, 512), (4, 4, 64, 8, 16, 0),
                 (3, 6, 64, 40, 1, 16), (256, 32, 128, 24, 64, 64)]:
        assert pa.decode_workspace_bytes(*args) == expect(*args), args
    # the partition length the call resolves: 0 asks for the default
    assert pa.decode_partition_tokens(0, 16, 512) == 1024  # table addresses 8192 tokens
    assert pa.decode_partition_tokens(0, 16, 256) == 1024  # 4096
    assert pa.decode_partition_tokens(0, 16, 255) == 512
    assert pa.decode_partition_tokens(0, 64, 24) == 512
    assert pa.decode_partition_tokens(768, 16, 512) == 768
    for bad in [(24, 16, 8), (-16, 16, 8), (0, 3, 8), (0, 16, 0), (64, 128, 8)]:
        with pytest.raises(pa.PagedAttnError):
            pa.decode_partition_tokens(*bad)
    # invalid sizes give 0
    assert pa.decode_workspace_bytes(4, 4, 96, 8, 16, 0) == 0
    assert pa.decode_workspace_bytes(4, 4, 64, 8, 3, 0) == 0
    assert pa.decode_workspace_bytes(4, 4, 64, 8, 16, 24) == 0


FAKE = 0x10000  # a 16-byte-aligned non-null address; never dereferenced by these calls


def _decode(lib, **kw):
    a = dict(out=FAKE, query=FAKE, kc=FAKE, vc=FAKE, bt=FAKE, sl=FAKE, S=2, Hq=8, Hkv=2, d=128,
             B=16, scale=0.1, MB=4, NB=100, pt=0, dtype=1, odt=None, ws=None, wsb=0)
    a.update(kw)
    return lib.pa_decode(a["out"], a["query"], a["kc"], a["vc"], a["bt"], a["sl"], a["S"], a["Hq"],
                         a["Hkv"], a["d"], a["B"], a["scale"], a["MB"], a["NB"], a["pt"], a["dtype"],
                         a["dtype"] if a["odt"] is None else a["odt"], a["ws"], a["wsb"], None)


@pytest.mark.parametrize("kw,code,msg", [
    (dict(dtype=5), -1, "dtype"),
    (dict(dtype=2), -1, "dtype"),
    (dict(odt=0), -1, "out_dtype"),
    (dict(S=-1), -1, "num_seqs"),
    (dict(Hq=6, Hkv=4), -1, "multiple"),
    (dict(Hq=34, Hkv=2), -2, "query heads per kv head"),
    (dict(d=96), -2, "head_dim"),
    (dict(B=12), -2, "block_size"),
    (dict(B=128), -2, "block_size"),
    (dict(MB=0), -1, "max_blocks_per_seq"),
    (dict(NB=0), -1, "num_blocks"),
    (dict(NB=1 << 27, B=64), -2, "slots"),           # 2^33 slots: above the 32-bit slot range
    (dict(scale=float("inf")), -1, "scale"),
    (dict(pt=24), -1, "partition_tokens"),
    (dict(pt=16, B=32), -1, "partition_tokens"),
    (dict(pt=1 << 21), -2, "partition_tokens"),
    (dict(out=None), -1, "NULL"),
    (dict(query=FAKE + 8), -1, "aligned"),
    (dict(bt=FAKE + 2), -1, "aligned"),
    (dict(MB=4096, pt=512), -3, "workspace"),
    (dict(MB=4096, pt=512, ws=FAKE, wsb=100), -3, "workspace"),
])
def test_decode_rejects_bad_arguments(lib, kw, code, msg):
    assert _decode(lib, **kw) == code
    assert msg in pa.last_error()


def test_decode_zero_sequences_is_a_no_op(lib):
    assert _decode(lib, S=0, out=None, query=None) == 0
    assert pa.last_error() == ""


def _write(lib, **kw):
    a = dict(k=FAKE, v=FAKE, kc=FAKE, vc=FAKE, slots=FAKE, T=3, Hkv=2, d=64, B=16, NB=10, dtype=0)
    a.update(kw)
    return lib.pa_reshape_and_cache(a["k"], a["v"], a["kc"], a["vc"], a["slots"], a["T"], a["Hkv"],
                                    a["d"], a["B"], a["NB"], a["dtype"], None)


@pytest.mark.parametrize("kw,code,msg", [
    (dict(dtype=3), -1, "dtype"),
    (dict(T=-2), -1, "num_tokens"),
    (dict(Hkv=0), -1, "num_kv_heads"),
    (dict(d=32), -2, "head_dim"),
    (dict(B=0), -2, "block_size"),
    (dict(NB=0), -1, "num_blocks"),
    (dict(kc=None), -1, "NULL"),
    (dict(k=FAKE + 4), -1, "aligned"),
    (dict(slots=FAKE + 4), -1, "aligned"),
])
def test_cache_write_rejects_bad_arguments(lib, kw, code, msg):
    assert _write(lib, **kw) == code
    assert msg in pa.last_error()


def test_cache_write_zero_tokens_is_a_no_op(lib):
    assert _write(lib, T=0, k=None) == 0


def _prefill(lib, **kw):
    a = dict(out=FAKE, query=FAKE, kc=FAKE, vc=FAKE, bt=FAKE, sl=FAKE, qs=FAKE, S=2, Hq=8, Hkv=2,
             d=128, B=16, scale=0.1, MB=4, NB=100, mq=64, dtype=1, odt=None, ws=None, wsb=0)
    a.update(kw)
    return lib.pa_prefill(a["out"], a["query"], a["kc"], a["vc"], a["bt"], a["sl"], a["qs"], a["S"],
                          a["Hq"], a["Hkv"], a["d"], a["B"], a["scale"], a["MB"], a["NB"], a["mq"],
                          a["dtype"], a["dtype"] if a["odt"] is None else a["odt"], a["ws"], a["wsb"],
                          None)


@pytest.mark.parametrize("kw,code,msg", [
    (dict(dtype=2), -1, "dtype"),
    (dict(odt=0), -1, "out_dtype"),
    (dict(S=-1), -1, "num_seqs"),
    (dict(Hq=6, Hkv=4), -1, "multiple"),
    (dict(Hq=34, Hkv=2), -2, "query heads per kv head"),
    (dict(d=256), -2, "head_dim"),
    (dict(B=3), -2, "block_size"),
    (dict(MB=0), -1, "max_blocks_per_seq"),
    (dict(NB=1 << 27, B=16), -2, "2^31"),
    (dict(scale=float("nan")), -1, "scale"),
    (dict(mq=-1), -1, "max_query_len"),
    (dict(qs=None), -1, "NULL"),
    (dict(out=FAKE + 8), -1, "aligned"),
    (dict(qs=FAKE + 2), -1, "aligned"),
    (dict(ws=FAKE, wsb=64), -3, "workspace"),
    (dict(ws=FAKE + 8, wsb=1 << 30), -1, "aligned"),
])
def test_prefill_rejects_bad_arguments(lib, kw, code, msg):
    assert _prefill(lib, **kw) == code
    assert msg in pa.last_error()


def test_prefill_workspace_bytes(lib):
    # bf16: an fp16 copy of every sequence's value rows, S * MB * B * Hkv * d * 2
    # bytes rounded up to 256; fp16 needs none; a copy of 2^31 slots or more is
    # not offered
    assert pa.prefill_workspace_bytes(16, 8, 128, 256, 16, "bf16") == 16 * 256 * 16 * 8 * 128 * 2
    assert pa.prefill_workspace_bytes(3, 1, 64, 5, 1, "bf16") == 2048  # 1920 rounded up
    assert pa.prefill_workspace_bytes(16, 8, 128, 256, 16, "fp16") == 0
    assert pa.prefill_workspace_bytes(4096, 8, 128, 1 << 16, 16, "bf16") == 0
    assert pa.prefill_workspace_bytes(4, 8, 96, 16, 16, "bf16") == 0
    # an fp16 call ignores a workspace it cannot use
    assert _prefill(lib, dtype=0, ws=FAKE, wsb=64, S=0, out=None) == 0


def test_prefill_empty_calls_are_no_ops(lib):
    assert _prefill(lib, S=0, out=None) == 0
    assert _prefill(lib, mq=0, out=None) == 0


def test_copy_blocks_rejects_bad_arguments(lib):
    assert lib.pa_copy_blocks(FAKE, FAKE, FAKE, FAKE, -1, 2, 128, 16, 10, 1, None) == -1
    assert lib.pa_copy_blocks(FAKE, FAKE, FAKE, FAKE, 1, 2, 80, 16, 10, 1, None) == -2
    assert lib.pa_copy_blocks(FAKE, FAKE, None, FAKE, 1, 2, 128, 16, 10, 1, None) == -1
    assert "NULL" in pa.last_error()
    assert lib.pa_copy_blocks(None, None, None, None, 0, 2, 128, 16, 10, 1, None) == 0


def test_wait_timeout_count_rejects_null(lib):
    assert lib.pa_wait_timeout_count(None, 0) == -1
    assert "NULL" in pa.last_error()


def test_bad_index_count_rejects_null(lib):
    assert lib.pa_bad_index_count(None, 0) == -1
    assert "NULL" in pa.last_error()


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(pa.pagedattn, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        pa.pagedattn.load_library(str(tmp_path / "libpagedattn.so"))
