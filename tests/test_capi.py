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
    fake = 1 << 20
    # one grid row per logit row: B * (D + 1) beyond 65535 is refused up front
    assert L.vc_accept(fake, 0, fake, 64, 1024, 8, fake, fake, fake, 1 << 30, None) == vc.VC_ERR_INVALID
    assert L.vc_accept_noalloc(fake, 0, fake, 1025, 0, 8, fake, fake, None) == vc.VC_ERR_INVALID
    assert L.vc_accept_noalloc(fake, 0, fake, 17, 1023, 8, fake, fake, None) == vc.VC_ERR_INVALID
    assert L.vc_workspace_init(None, 0, None) == vc.VC_ERR_INVALID


def test_decoder_validation_on_the_host(libvc):
    """vc_decoder_create checks the configuration and the weight pointers and
    allocates nothing; unsupported shapes are refused, not approximated."""
    import ctypes
    from lossless_draft_verify_gb300 import vc
    L = vc.load()
    n = 2
    arr = ctypes.c_void_p * n
    ptrs = [arr(*[4096 * (i + 1 + 16 * k) for i in range(n)]) for k in range(4)]
    w = vc.DecoderWeights(1 << 20, 2 << 20, *ptrs)
    h = ctypes.c_void_p()

    def create(**kw):
        base = dict(n_layers=n, d_model=256, n_heads=4, n_kv_heads=2, head_dim=64, d_ff=512, vocab=512,
                    norm_eps=1e-6, rope_theta=1e4, dt=vc.VC_F32)
        base.update(kw)
        c = vc.DecoderCfg(**base)
        return L.vc_decoder_create(ctypes.byref(c), ctypes.byref(w), ctypes.byref(h))

    assert create() == vc.VC_OK and h.value
    assert L.vc_decoder_workspace_bytes(h, 1, 16, 1024, None) > 0
    assert L.vc_decoder_workspace_bytes(h, 0, 16, 1024, None) == 0
    # per-layer arrival events: one non-null handle per layer, or none
    evs = (ctypes.c_void_p * n)(0x1000, 0x2000)
    assert L.vc_decoder_set_layer_events(h, evs, n) == vc.VC_OK
    assert L.vc_decoder_set_layer_events(h, None, 0) == vc.VC_OK
    assert L.vc_decoder_set_layer_events(h, evs, n - 1) == vc.VC_ERR_INVALID
    assert L.vc_decoder_set_layer_events(h, None, n) == vc.VC_ERR_INVALID
    assert L.vc_decoder_set_layer_events(h, (ctypes.c_void_p * n)(0x1000, None), n) == vc.VC_ERR_INVALID
    assert L.vc_decoder_set_layer_events(h, evs, -1) == vc.VC_ERR_INVALID
    assert L.vc_decoder_set_layer_events(None, evs, n) == vc.VC_ERR_INVALID
    L.vc_decoder_destroy(h)
    assert create(head_dim=96) == vc.VC_ERR_UNSUPPORTED
    assert create(n_heads=16, n_kv_heads=2) == vc.VC_ERR_UNSUPPORTED     # 8 q heads per kv head
    assert create(n_heads=6, n_kv_heads=4) == vc.VC_ERR_UNSUPPORTED
    assert create(n_layers=0) == vc.VC_ERR_INVALID
    assert create(dt=7) == vc.VC_ERR_INVALID
    bad = vc.DecoderWeights(None, 2 << 20, *ptrs)
    c = vc.DecoderCfg(n, 256, 4, 2, 64, 512, 512, 1e-6, 1e4, vc.VC_F32)
    assert L.vc_decoder_create(ctypes.byref(c), ctypes.byref(bad), ctypes.byref(h)) == vc.VC_ERR_INVALID
    assert L.vc_decoder_forward(None, None, None, 0, 1, 1, None, 0, None, None, 1, None, None, 0, None, None, 0,
                                None) == vc.VC_ERR_INVALID
    assert L.vc_gemm(None, None, None, None, 0, 1, 1, 1, None, 0, None) == vc.VC_ERR_INVALID
    assert L.vc_kv_writeback(None, None, 0, 1, 1, 1, 1, 64, None, None, None, None, 8, None) == vc.VC_ERR_INVALID


def test_greedy_head_and_rotation_validation_on_the_host(libvc):
    """The argmax-epilogue GEMM, acceptance from tile maxima, the fused verify
    call and the rotated-cache flag reject bad arguments before any CUDA call."""
    import ctypes
    from lossless_draft_verify_gb300 import vc
    L = vc.load()
    fake = 1 << 20                      # aligned, never dereferenced on these paths
    # argmax epilogue: null pointers; shapes or types without a tensor-core head
    assert L.vc_gemm_argmax(None, fake, vc.VC_BF16, 8, 256, 64, 0, fake, fake, None, 0, None) == vc.VC_ERR_INVALID
    assert L.vc_gemm_argmax(fake, fake, vc.VC_F32, 8, 256, 64, 0, fake, fake, None, 0,
                            None) == vc.VC_ERR_UNSUPPORTED
    assert L.vc_gemm_argmax(fake, fake, vc.VC_BF16, 8, 200, 64, 0, fake, fake, None, 0,
                            None) == vc.VC_ERR_UNSUPPORTED              # N not a multiple of 128
    assert L.vc_gemm_argmax(fake, fake, vc.VC_BF16, 8, 256, 40, 0, fake, fake, None, 0,
                            None) == vc.VC_ERR_UNSUPPORTED              # K not a multiple of 64
    # acceptance from tile maxima
    assert L.vc_accept_tiles(None, fake, 4, fake, 2, 3, fake, fake, None) == vc.VC_ERR_INVALID
    assert L.vc_accept_tiles(fake, fake, 0, fake, 2, 3, fake, fake, None) == vc.VC_ERR_INVALID
    assert L.vc_accept_tiles(fake, fake, 4, None, 2, 3, fake, fake, None) == vc.VC_ERR_INVALID   # D > 0 needs drafts
    assert L.vc_accept_tiles(fake, fake, 4, fake, 2, 1025, fake, fake, None) == vc.VC_ERR_INVALID
    # fused verify: no decoder
    assert L.vc_decoder_verify(None, fake, fake, 4, 2, fake, 0, fake, fake, 8, None, None, fake, fake, fake, 1 << 20,
                               None) == vc.VC_ERR_INVALID
    # the rotated-cache flag takes 0 or 1
    q = vc.QCacheC(fake, fake, fake, fake, fake, fake, 1, 1, 128, vc.QuantCfg(2, 32, 0, 2), 4, 64, vc.VC_BF16)
    assert L.vc_quantize_kv(fake, fake, vc.VC_BF16, 1, 1, 32, 32, 128, ctypes.byref(q), None) == vc.VC_ERR_INVALID


def test_normalised_row_gemm_validation_on_the_host(libvc):
    """vc_gemm_rms (the draft steps' products of RMS-normalised rows) rejects
    bad arguments and shapes outside its path before any CUDA call."""
    from lossless_draft_verify_gb300 import vc
    L = vc.load()
    fake = 1 << 20                      # aligned, never dereferenced on these paths
    ok_args = (fake, fake, fake, vc.VC_BF16, 8, 4096, 4096)
    assert L.vc_gemm_rms(None, fake, fake, vc.VC_BF16, 8, 4096, 4096, 1e-5, 0, None, 0, None) == vc.VC_ERR_INVALID
    assert L.vc_gemm_rms(*ok_args, -1.0, 0, None, 0, None) == vc.VC_ERR_INVALID          # eps < 0
    assert L.vc_gemm_rms(*ok_args, float("nan"), 0, None, 0, None) == vc.VC_ERR_INVALID
    assert L.vc_gemm_rms(fake + 2, fake, fake, vc.VC_BF16, 8, 4096, 4096, 1e-5, 0, None, 0,
                         None) == vc.VC_ERR_INVALID                                    # x not 16-byte aligned
    assert L.vc_gemm_rms(fake, fake, fake, vc.VC_BF16, 17, 4096, 4096, 1e-5, 0, None, 0,
                         None) == vc.VC_ERR_UNSUPPORTED                                # more than 16 rows
    assert L.vc_gemm_rms(fake, fake, fake, vc.VC_F32, 8, 4096, 4096, 1e-5, 0, None, 0,
                         None) == vc.VC_ERR_UNSUPPORTED
    assert L.vc_gemm_rms(fake, fake, fake, vc.VC_BF16, 8, 4000, 4096, 1e-5, 0, None, 0,
                         None) == vc.VC_ERR_UNSUPPORTED                                # N not a multiple of 128
    assert L.vc_gemm_rms(fake, fake, fake, vc.VC_BF16, 8, 2048, 1024, 1e-5, 1, None, 0,
                         None) == vc.VC_ERR_UNSUPPORTED                                # SwiGLU of a split product
    # a split product needs its workspace
    assert L.vc_gemm_rms(*ok_args, 1e-5, 0, None, 0, None) == vc.VC_ERR_INVALID


def test_kv_pack_validation_on_the_host(libvc):
    """Packing and unpacking reject bad arguments before any CUDA call; zero
    rows are a no-op."""
    from lossless_draft_verify_gb300 import vc
    L = vc.load()
    fake = 1 << 20
    assert L.vc_kv_packed_row_bytes(128) == 208 and L.vc_kv_packed_row_bytes(64) == 112
    assert L.vc_kv_packed_row_bytes(96) == 0
    assert L.vc_kv_pack(None, fake, 4, 128, None, None) == vc.VC_ERR_INVALID
    assert L.vc_kv_pack(fake, fake, -1, 128, None, None) == vc.VC_ERR_INVALID
    assert L.vc_kv_pack(fake, fake, 4, 96, None, None) == vc.VC_ERR_UNSUPPORTED
    assert L.vc_kv_pack(fake + 4, fake, 4, 128, None, None) == vc.VC_ERR_INVALID     # source not 8-byte aligned
    assert L.vc_kv_pack(fake, fake + 8, 4, 128, None, None) == vc.VC_ERR_INVALID     # rows not 16-byte aligned
    assert L.vc_kv_pack(None, None, 0, 128, None, None) == vc.VC_OK
    assert L.vc_kv_unpack(fake, None, 4, 64, None) == vc.VC_ERR_INVALID
    assert L.vc_kv_unpack(fake + 8, fake, 4, 64, None) == vc.VC_ERR_INVALID
    assert L.vc_kv_unpack(fake, fake, 4, 32, None) == vc.VC_ERR_UNSUPPORTED
    assert L.vc_kv_unpack(None, None, 0, 64, None) == vc.VC_OK


def test_kv_packed_row_size_agrees_with_the_oracle(libvc):
    """The library's packed row size and the oracle's format give the same
    bytes per row (both stated independently)."""
    import oracle
    from lossless_draft_verify_gb300 import vc
    L = vc.load()
    for d in (64, 128):
        assert L.vc_kv_packed_row_bytes(d) == oracle.kv_packed_row_bytes(d)
