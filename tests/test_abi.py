"""The C-ABI library builds, loads and exports every declared entry point; host-side
validation rejects bad arguments before any CUDA call. No test here needs a GPU."""
import ctypes
import os
import re

import pytest

from paged_decode_attention_02_gb300 import binding, build_lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pda.h")


@pytest.fixture(scope="module")
def lib():
    build_lib.build()
    return binding.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pda_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding_names():
    assert declared_functions() == sorted(binding.EXPORTED)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_version_and_status_strings(lib):
    assert lib.pda_version() == 1
    assert binding.status_string(0) == "ok"
    for s in range(1, 5):
        assert binding.status_string(s) not in ("ok", "unknown status")
    assert binding.status_string(99) == "unknown status"


FAKE = ctypes.c_void_p(1 << 20)  # aligned, never dereferenced: every call below fails first


def _attn(lib, **kw):
    a = dict(out=FAKE, q=FAKE, k=FAKE, v=FAKE, bt=FAKE, max_blocks=4, cl=FAKE, max_ctx=64, B=2,
             H=4, H_kv=2, D=128, bs=16, NB=8, scale=0.1, qd=1, kvd=1, od=1, cap=0, ws=FAKE,
             ws_bytes=1 << 20, err=None, stream=None)
    a.update(kw)
    return lib.pda_paged_decode_attention(a["out"], a["q"], a["k"], a["v"], a["bt"],
                                          a["max_blocks"], a["cl"], a["max_ctx"], a["B"], a["H"],
                                          a["H_kv"], a["D"], a["bs"], a["NB"], a["scale"],
                                          a["qd"], a["kvd"], a["od"], a["cap"], a["ws"],
                                          a["ws_bytes"], a["err"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(H=5), binding.PDA_ERR_INVALID_ARG),            # H % H_kv != 0
    (dict(B=-1), binding.PDA_ERR_INVALID_ARG),
    (dict(q=None), binding.PDA_ERR_INVALID_ARG),
    (dict(kvd=7), binding.PDA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), binding.PDA_ERR_INVALID_ARG),
    (dict(out=ctypes.c_void_p((1 << 20) + 4)), binding.PDA_ERR_INVALID_ARG),  # misaligned
    (dict(D=96), binding.PDA_ERR_UNSUPPORTED),
    (dict(bs=24), binding.PDA_ERR_UNSUPPORTED),          # not a multiple of the 16-row tile
    (dict(bs=8), binding.PDA_ERR_UNSUPPORTED),
    (dict(bs=48), binding.PDA_ERR_UNSUPPORTED),          # not a power of two
    (dict(bs=512), binding.PDA_ERR_UNSUPPORTED),
    (dict(H=24, H_kv=2), binding.PDA_ERR_UNSUPPORTED),   # group of 12
    (dict(qd=0), binding.PDA_ERR_UNSUPPORTED),           # q dtype != kv dtype
    (dict(B=9000), binding.PDA_ERR_UNSUPPORTED),
    (dict(ws=None), binding.PDA_ERR_WORKSPACE),
    (dict(ws=ctypes.c_void_p((1 << 20) + 16)), binding.PDA_ERR_WORKSPACE),
])
def test_attention_rejects_bad_arguments(lib, kw, status):
    assert _attn(lib, **kw) == status


def test_attention_empty_batch_is_noop(lib):
    assert _attn(lib, B=0, q=None, out=None) == binding.PDA_OK


def test_append_and_pack_reject_bad_arguments(lib):
    f = lib.pda_kv_append
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, -1, 2, 64, 16, 8, 1, None, None) == 1
    assert f(None, FAKE, FAKE, FAKE, FAKE, 3, 2, 64, 16, 8, 1, None, None) == 1
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 3, 1, 4, 16, 8, 1, None, None) == 2  # 8-byte rows
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 2, 64, 16, 8, 1, None, None) == 0
    g = lib.pda_kv_pack_blocks
    assert g(FAKE, FAKE, FAKE, FAKE, -1, 2, 64, 16, 8, 1, None, None) == 1
    assert g(FAKE, FAKE, FAKE, FAKE, 0, 2, 64, 16, 8, 1, None, None) == 0
    assert g(None, FAKE, FAKE, FAKE, 5, 2, 64, 16, 8, 1, None, None) == 1
    h = lib.pda_kv_pack_blocks_batched
    assert h(None, None, None, 65, FAKE, FAKE, 2, 64, 16, 8, 1, None, None) == 2


def test_workspace_query_validates_before_touching_the_device(lib):
    n = ctypes.c_size_t(0)
    assert lib.pda_attention_workspace_size(4, 4, 3, 128, 16, 1, 0, ctypes.byref(n)) == 1
    assert lib.pda_attention_workspace_size(4, 4, 2, 80, 16, 1, 0, ctypes.byref(n)) == 2
    assert lib.pda_attention_workspace_size(4, 4, 2, 128, 16, 1, 0, None) == 1
