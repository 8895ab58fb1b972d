"""CPU checks of the C-ABI library: it builds, loads without a GPU, exports
every entry point that include/vc.h declares, and its pure host helpers
(status strings, record size, kept-token count) behave as documented."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "vc.h")


def _declared():
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(vc_\w+)\s*\(", txt)))


@pytest.fixture(scope="module")
def libvc():
    from lossless_draft_verify_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("vc_quantize_kv", "vc_drop_tokens", "vc_draft_attn", "vc_verify_attn", "vc_accept",
              "vc_swap_in"):
        assert n in names


def test_library_exports_every_declared_symbol(libvc):
    missing = [n for n in _declared() if not hasattr(libvc, n)]
    assert not missing, missing


def test_binding_covers_every_export():
    from lossless_draft_verify_gb300 import vc
    assert sorted(vc.EXPORTED) == _declared()


def test_host_helpers(libvc):
    from lossless_draft_verify_gb300 import vc
    vc.load()
    assert vc.status_str(0) == "ok"
    assert "invalid" in vc.status_str(1)
    assert vc.vc_record_bytes(2, 128) == 3072 and vc.vc_record_bytes(4, 64) == 2560
    assert vc.vc_record_bytes(3, 128) == 0
    assert vc.vc_drop_kept_count(131072, 32768, 256) == 33024
    assert vc.vc_drop_kept_count(100, 500, 30) == 100
    assert vc.vc_drop_kept_count(10, 3, 50) == 10
    assert "sm_103a" in vc.vc_version()


def test_invalid_arguments_are_rejected_on_the_host(libvc):
    """Null pointers and bad sizes return VC_ERR_INVALID before any CUDA call."""
    from lossless_draft_verify_gb300 import vc
    L = vc.load()
    assert L.vc_accept(None, 0, None, 1, 0, 10, None, None, None, 0, None) == vc.VC_ERR_INVALID
    assert L.vc_verify_attn(None, None, None, 0, None, 1, 1, 4, 2, 128, 64, 0, 1.0, None, None, 0,
                            None) == vc.VC_ERR_INVALID
    assert L.vc_swap_in(None, None, 16, None, None) == vc.VC_ERR_INVALID
    assert L.vc_workspace_init(None, 0, None) == vc.VC_ERR_INVALID
