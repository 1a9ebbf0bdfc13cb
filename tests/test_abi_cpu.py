"""CPU-only checks of the C-ABI library: it builds for sm_103a, loads, exports
every entry point include/compkv.h declares, and validates arguments on the
host (no compute call needs a GPU here).  Also checks that the oracle and the
product path share no code."""
import ctypes
import os
import re
import subprocess

import pytest

import block_sparse_kv_summary_gb300 as P
from block_sparse_kv_summary_gb300 import compkv as C

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    P.build()
    return P.lib()


def header_functions():
    src = open(os.path.join(ROOT, "include", "compkv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(compkv_\w+)\s*\(", src)))


def test_header_declares_the_calls():
    names = header_functions()
    for n in ("compkv_init", "compkv_append", "compkv_score_select", "compkv_attend", "compkv_decode",
              "compkv_device_status", "compkv_destroy", "compkv_prefill", "compkv_scratch_bytes"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    names = header_functions()
    out = subprocess.run(["nm", "-D", "--defined-only", P.library_file], capture_output=True, text=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if line.strip())
    missing = [n for n in names if n not in exported]
    assert not missing, f"not exported: {missing}"
    for n in names:
        assert hasattr(lib, n)
        assert hasattr(C, n), f"binding lacks {n}"


def test_build_targets_sm103a_only():
    from block_sparse_kv_summary_gb300 import _build
    assert _build.ARCH == "-gencode=arch=compute_103a,code=sm_103a"
    assert _build.ARCH in _build.NVCC_FLAGS


def cfg(**kw):
    base = dict(num_layers=1, batch=2, num_kv_heads=8, group_size=4, head_dim=128, r=4,
                budget_tokens=2048, max_tokens=131136)
    base.update(kw)
    return C.make_config(**base)


@pytest.mark.parametrize("bad,msg", [
    (dict(group_size=3), "group_size"),
    (dict(head_dim=96), "head_dim"),
    (dict(r=3), "r must"),
    (dict(r=256), "r must"),
    (dict(budget_tokens=100), "budget_tokens"),
    (dict(budget_tokens=32), "budget_tokens"),
    (dict(batch=0), "batch"),
    (dict(batch=65), "batch"),
    (dict(num_kv_heads=33), "num_kv_heads"),
    (dict(max_tokens=100), "capacity"),
    (dict(max_tokens=16 * 140000), "does not fit"),
    (dict(variant=8), "variant"),
])
def test_config_validation(lib, bad, msg):
    c = cfg(**bad)
    assert C.compkv_scratch_bytes(c) == 0
    assert msg in C.compkv_last_error()
    bufs = C.compkv_buffers(16, 16, 16, 16, 16, 16, 256, 1 << 30)
    with pytest.raises(C.CompKVError) as e:
        C.compkv_init(c, bufs)
    assert e.value.status in (1, 2)


def test_block_size_must_be_16(lib):
    c = cfg()
    c.block_size = 32
    assert C.compkv_scratch_bytes(c) == 0


def test_init_rejects_bad_buffers(lib):
    c = cfg()
    need = C.compkv_scratch_bytes(c)
    with pytest.raises(C.CompKVError, match="scratch_bytes"):
        C.compkv_init(c, C.compkv_buffers(256, 256, 256, 256, 256, 256, 256, need - 1))
    with pytest.raises(C.CompKVError, match="k is NULL"):
        C.compkv_init(c, C.compkv_buffers(0, 256, 256, 256, 256, 256, 256, need))
    with pytest.raises(C.CompKVError, match="aligned"):
        C.compkv_init(c, C.compkv_buffers(258, 256, 256, 256, 256, 256, 256, need))


def test_ragged_rows_and_scratch(lib):
    caps = [8208, 131088, 32784]
    c = cfg(batch=3, capacity_tokens=caps)
    assert C.compkv_rows_per_layer(c) == 8 * sum(x // 16 for x in caps)
    uni = cfg(batch=3, max_tokens=131088)
    assert C.compkv_scratch_bytes(c) < C.compkv_scratch_bytes(uni)
    assert C.compkv_scratch_bytes(c) % 256 == 0


def test_calls_reject_null_context(lib):
    assert lib.compkv_append(None, 0, None, None, None) == 1
    assert lib.compkv_decode(None, 0, None, None, None, None, None, None) == 1
    assert lib.compkv_device_status(None, None) == 1
    assert lib.compkv_launch_count(None) == 0
    assert C.compkv_status_string(6) == "COMPKV_ERR_BAD_SELECTION"


def _imports(path):
    pat = re.compile(r"^\s*(?:from|import)\s+([\w\.]+)", re.M)
    found = set()
    for dp, _, files in os.walk(path):
        for f in files:
            if f.endswith(".py"):
                found |= set(m.split(".")[0] for m in pat.findall(open(os.path.join(dp, f)).read()))
    return found


def test_oracle_and_product_share_nothing():
    assert "block_sparse_kv_summary_gb300" not in _imports(os.path.join(ROOT, "oracle"))
    assert "oracle" not in _imports(os.path.join(ROOT, "block_sparse_kv_summary_gb300"))
    assert "oracle" not in _imports(os.path.join(ROOT, "synth"))
    csrc = os.path.join(ROOT, "block_sparse_kv_summary_gb300", "csrc")
    for f in os.listdir(csrc):
        assert "oracle" not in open(os.path.join(csrc, f)).read().lower()


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(C, "_lib", None)
    monkeypatch.setattr(C, "LIB", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        C.lib()
