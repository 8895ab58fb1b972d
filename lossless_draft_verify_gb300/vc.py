"""Thin Python binding of the C ABI in include/vc.h (ctypes).

Argument marshalling only: every function here turns torch tensors into
pointers and sizes, calls the entry point of the same name in libvc.so and
raises on a non-OK status.  No computation happens in Python, and there is no
fallback: if the library is missing or cannot be loaded, importing the
functions raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libvc.so")

VC_OK, VC_ERR_INVALID, VC_ERR_UNSUPPORTED, VC_ERR_CUDA, VC_ERR_TIMEOUT = 0, 1, 2, 3, 4
VC_BF16, VC_F32 = 0, 1
VC_CACHE_KIVI, VC_CACHE_DENSE = 0, 1

c_void_p, c_int, c_float, c_size_t, c_int64 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_float,
                                                ctypes.c_size_t, ctypes.c_int64)
c_int32 = ctypes.c_int32


class VcError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_str(status)} (status {status})")


class QuantCfg(ctypes.Structure):
    _fields_ = [("bits", c_int32), ("group", c_int32), ("residual", c_int32), ("rotate", c_int32)]


class QCacheC(ctypes.Structure):
    _fields_ = [("records", c_void_p), ("k_res", c_void_p), ("v_res", c_void_p),
                ("n_groups", c_void_p), ("seq_len", c_void_p), ("status", c_void_p),
                ("B", c_int32), ("Hkv", c_int32), ("d", c_int32), ("cfg", QuantCfg),
                ("max_groups", c_int32), ("res_cap", c_int32), ("res_dtype", c_int)]


class DropCfg(ctypes.Structure):
    _fields_ = [("keep_top", c_int64), ("keep_recent", c_int64)]


class CacheView(ctypes.Structure):
    _fields_ = [("kind", c_int), ("kivi", ctypes.POINTER(QCacheC)), ("k", c_void_p), ("v", c_void_p),
                ("dt", c_int), ("seq_len", c_void_p), ("B", c_int32), ("Hkv", c_int32), ("d", c_int32),
                ("L_stride", c_int32), ("max_len", c_int32), ("flags", c_int32)]


class DecoderCfg(ctypes.Structure):
    _fields_ = [("n_layers", c_int32), ("d_model", c_int32), ("n_heads", c_int32), ("n_kv_heads", c_int32),
                ("head_dim", c_int32), ("d_ff", c_int32), ("vocab", c_int32), ("norm_eps", c_float),
                ("rope_theta", c_float), ("dt", c_int)]


class DecoderWeights(ctypes.Structure):
    _fields_ = [("embed", c_void_p), ("lm_head", c_void_p), ("w_qkv", ctypes.POINTER(c_void_p)),
                ("w_o", ctypes.POINTER(c_void_p)), ("w_gate_up", ctypes.POINTER(c_void_p)),
                ("w_down", ctypes.POINTER(c_void_p))]


_lib = None


def load() -> ctypes.CDLL:
    """Load libvc.so (built by lossless_draft_verify_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libvc.so not built ({LIB_PATH}); run lossless_draft_verify_gb300.build.build()")
    L = ctypes.CDLL(LIB_PATH)
    P = c_void_p
    L.vc_status_str.restype = ctypes.c_char_p
    L.vc_status_str.argtypes = [c_int]
    L.vc_version.restype = ctypes.c_char_p
    L.vc_check.restype = c_int
    L.vc_check.argtypes = [P]
    L.vc_workspace_init.restype = c_int
    L.vc_workspace_init.argtypes = [P, c_size_t, P]
    L.vc_poll_status.restype = c_int
    L.vc_poll_status.argtypes = [P, P]
    L.vc_record_bytes.restype = c_size_t
    L.vc_record_bytes.argtypes = [c_int, c_int]
    L.vc_quantize_kv.restype = c_int
    L.vc_quantize_kv.argtypes = [P, P, c_int, c_int, c_int, c_int, c_int, c_int, ctypes.POINTER(QCacheC), P]
    L.vc_qcache_append.restype = c_int
    L.vc_qcache_append.argtypes = [ctypes.POINTER(QCacheC), P, P, P, c_int, c_int, P]
    L.vc_qcache_commit.restype = c_int
    L.vc_qcache_commit.argtypes = [ctypes.POINTER(QCacheC), P, P, P, P, c_int, P]
    L.vc_drop_kept_count.restype = c_int64
    L.vc_drop_kept_count.argtypes = [c_int64, DropCfg]
    L.vc_drop_tokens_workspace_bytes.restype = c_size_t
    L.vc_drop_tokens_workspace_bytes.argtypes = [c_int, c_int, c_int]
    L.vc_drop_tokens.restype = c_int
    L.vc_drop_tokens.argtypes = [P, P, P, c_int, c_int, c_int, c_int, c_int, DropCfg, P, P, P, P, c_size_t, P]
    L.vc_draft_attn_workspace_bytes.restype = c_size_t
    L.vc_draft_attn_workspace_bytes.argtypes = [ctypes.POINTER(CacheView), c_int]
    L.vc_draft_attn.restype = c_int
    L.vc_draft_attn.argtypes = [P, c_int, ctypes.POINTER(CacheView), c_int, c_float, P, P, c_size_t, P]
    L.vc_draft_attn_h2o_workspace_bytes.restype = c_size_t
    L.vc_draft_attn_h2o_workspace_bytes.argtypes = [ctypes.POINTER(CacheView), c_int]
    L.vc_draft_attn_h2o.restype = c_int
    L.vc_draft_attn_h2o.argtypes = [P, c_int, ctypes.POINTER(CacheView), c_int, c_float, P, P, c_int, P, c_int, P,
                                    c_size_t, P]
    L.vc_verify_attn_workspace_bytes.restype = c_size_t
    L.vc_verify_attn_workspace_bytes.argtypes = [c_int, c_int, c_int, c_int, c_int, c_int, c_int]
    L.vc_verify_attn.restype = c_int
    L.vc_verify_attn.argtypes = [P, P, P, c_int, P, c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_float,
                                 P, P, c_size_t, P]
    L.vc_verify_attn_h2o_workspace_bytes.restype = c_size_t
    L.vc_verify_attn_h2o_workspace_bytes.argtypes = [c_int, c_int, c_int, c_int, c_int, c_int]
    L.vc_verify_attn_h2o.restype = c_int
    L.vc_verify_attn_h2o.argtypes = [P, P, P, P, c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_float, P, P,
                                     c_int, P, c_size_t, P]
    L.vc_accept_workspace_bytes.restype = c_size_t
    L.vc_accept_workspace_bytes.argtypes = [c_int, c_int, c_int]
    L.vc_accept.restype = c_int
    L.vc_accept.argtypes = [P, c_int, P, c_int, c_int, c_int, P, P, P, c_size_t, P]
    L.vc_accept_noalloc.restype = c_int
    L.vc_accept_noalloc.argtypes = [P, c_int, P, c_int, c_int, c_int, P, P, P]
    L.vc_wait_probe.restype = c_int
    L.vc_wait_probe.argtypes = [P, c_size_t, P]
    L.vc_swap_in_paced.restype = c_int
    L.vc_swap_in_paced.argtypes = [P, P, c_size_t, ctypes.c_double, c_size_t, P, P, P]
    L.vc_swap_in.restype = c_int
    L.vc_swap_in.argtypes = [P, P, c_size_t, P, P]
    L.vc_decoder_create.restype = c_int
    L.vc_decoder_create.argtypes = [ctypes.POINTER(DecoderCfg), ctypes.POINTER(DecoderWeights),
                                    ctypes.POINTER(c_void_p)]
    L.vc_decoder_destroy.restype = None
    L.vc_decoder_destroy.argtypes = [P]
    L.vc_decoder_workspace_bytes.restype = c_size_t
    L.vc_decoder_workspace_bytes.argtypes = [P, c_int, c_int, c_int, ctypes.POINTER(QCacheC)]
    L.vc_decoder_forward.restype = c_int
    L.vc_decoder_forward.argtypes = [P, P, P, c_int, c_int, c_int, P, c_int, P, P, c_int, P, P, c_int, P, P,
                                     c_size_t, P]
    L.vc_decoder_draft_step.restype = c_int
    L.vc_decoder_draft_step.argtypes = [P, P, c_int, ctypes.POINTER(QCacheC), P, P, P, c_int, P, c_size_t, P]
    L.vc_kv_writeback.restype = c_int
    L.vc_kv_writeback.argtypes = [P, P, c_int, c_int, c_int, c_int, c_int, c_int, P, P, P, P, c_int, P]
    L.vc_decoder_set_trace.restype = c_int
    L.vc_decoder_set_trace.argtypes = [P, P, P, c_int, c_int]
    L.vc_decoder_trace_count.restype = c_int
    L.vc_decoder_trace_count.argtypes = [P]
    L.vc_decoder_set_layer_events.restype = c_int
    L.vc_decoder_set_layer_events.argtypes = [P, P, c_int]
    L.vc_gemm_splits.restype = c_int
    L.vc_gemm_splits.argtypes = [c_int, c_int, c_int, c_int]
    L.vc_gemm_workspace_bytes.restype = c_size_t
    L.vc_gemm_workspace_bytes.argtypes = [c_int, c_int, c_int, c_int]
    L.vc_gemm.restype = c_int
    L.vc_gemm.argtypes = [P, P, P, P, c_int, c_int, c_int, c_int, P, c_size_t, P]
    L.vc_gemm_ex.restype = c_int
    L.vc_gemm_ex.argtypes = [P, P, P, P, c_int, c_int, c_int, c_int, c_int, P, c_size_t, P]
    L.vc_gemm_argmax.restype = c_int
    L.vc_gemm_argmax.argtypes = [P, P, c_int, c_int, c_int, c_int, c_int, P, P, P, c_size_t, P]
    L.vc_gemm_swiglu.restype = c_int
    L.vc_gemm_rms.restype = c_int
    L.vc_gemm_rms.argtypes = [P, P, P, c_int, c_int, c_int, c_int, ctypes.c_float, c_int, P, c_size_t, P]
    L.vc_swap_in_rows.restype = c_int
    L.vc_swap_in_rows.argtypes = [P, P, c_size_t, c_size_t, c_size_t, c_size_t, P, P]
    L.vc_gemm_swiglu.argtypes = [P, P, P, c_int, c_int, c_int, c_int, c_int, P]
    L.vc_accept_tiles.restype = c_int
    L.vc_accept_tiles.argtypes = [P, P, c_int, P, c_int, c_int, P, P, P]
    L.vc_decoder_verify.restype = c_int
    L.vc_decoder_verify.argtypes = [P, P, P, c_int, c_int, P, c_int, P, P, c_int, P, P, P, P, P, c_size_t, P]
    L.vc_kv_packed_row_bytes.restype = c_size_t
    L.vc_kv_packed_row_bytes.argtypes = [c_int]
    L.vc_kv_pack.restype = c_int
    L.vc_kv_pack.argtypes = [P, P, c_int64, c_int, P, P]
    L.vc_kv_unpack.restype = c_int
    L.vc_kv_unpack.argtypes = [P, P, c_int64, c_int, P]
    L.vc_kv_writeback_packed.restype = c_int
    L.vc_kv_writeback_packed.argtypes = [P, P, c_int, c_int, c_int, c_int, c_int, P, P, P, P, c_int, P, P]
    _lib = L
    return L


EXPORTED = ["vc_status_str", "vc_version", "vc_check", "vc_workspace_init", "vc_poll_status",
            "vc_record_bytes", "vc_quantize_kv", "vc_qcache_append", "vc_qcache_commit", "vc_drop_kept_count",
            "vc_drop_tokens_workspace_bytes", "vc_drop_tokens", "vc_draft_attn_workspace_bytes",
            "vc_draft_attn", "vc_verify_attn_workspace_bytes", "vc_verify_attn",
            "vc_accept_workspace_bytes", "vc_accept", "vc_accept_noalloc", "vc_swap_in",
            "vc_decoder_create", "vc_decoder_destroy", "vc_decoder_workspace_bytes", "vc_decoder_forward",
            "vc_decoder_draft_step", "vc_kv_writeback", "vc_gemm_workspace_bytes", "vc_gemm",
            "vc_decoder_set_trace", "vc_decoder_trace_count", "vc_gemm_splits",
            "vc_draft_attn_h2o_workspace_bytes", "vc_draft_attn_h2o", "vc_gemm_ex", "vc_wait_probe",
            "vc_swap_in_paced", "vc_gemm_argmax", "vc_accept_tiles", "vc_decoder_verify",
            "vc_kv_packed_row_bytes", "vc_kv_pack", "vc_kv_unpack", "vc_kv_writeback_packed",
            "vc_verify_attn_h2o_workspace_bytes", "vc_verify_attn_h2o", "vc_decoder_set_layer_events",
            "vc_gemm_swiglu", "vc_swap_in_rows", "vc_gemm_rms"]

TRACE_KINDS = ["gemm_qkv", "gemm_o", "gemm_gate_up", "gemm_down", "gemm_head", "draft_attn", "verify_attn"]


def status_str(s: int) -> str:
    return load().vc_status_str(int(s)).decode()


def _check(rc: int, where: str):
    if rc != VC_OK:
        raise VcError(rc, where)


def _ptr(t) -> int:
    if t is None:
        return None
    return t.data_ptr()


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return VC_BF16
    if t.dtype == torch.float32:
        return VC_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _stream(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


# ---------------------------------------------------------------- memory --

class Workspace:
    """A zero-initialised device workspace (the caller-owned scratch buffer)."""

    def __init__(self, nbytes: int, device="cuda"):
        self.nbytes = max(int(nbytes), 256)
        self.buf = torch.zeros(self.nbytes, dtype=torch.uint8, device=device)

    def ensure(self, nbytes: int):
        if nbytes > self.nbytes:
            self.__init__(nbytes, self.buf.device)
        return self

    @property
    def ptr(self):
        return self.buf.data_ptr()


class QCache:
    """Caller-owned storage of one layer's KIVI cache (include/vc.h, vc_qcache)."""

    def __init__(self, B, Hkv, d, bits, max_groups, res_cap, residual=0, group=32,
                 res_dtype=torch.bfloat16, device="cuda", rotate: bool = False):
        rb = vc_record_bytes(bits, d)
        self.rec_bytes = rb
        self.records = torch.zeros(B * Hkv * max(max_groups, 1) * rb, dtype=torch.uint8, device=device)
        self.k_res = torch.zeros(B, Hkv, res_cap, d, dtype=res_dtype, device=device)
        self.v_res = torch.zeros_like(self.k_res)
        self.n_groups = torch.zeros(B, dtype=torch.int32, device=device)
        self.seq_len = torch.zeros(B, dtype=torch.int32, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.c = QCacheC(self.records.data_ptr(), self.k_res.data_ptr(), self.v_res.data_ptr(),
                         self.n_groups.data_ptr(), self.seq_len.data_ptr(), self.status.data_ptr(),
                         B, Hkv, d, QuantCfg(bits, group, residual, int(bool(rotate))), max_groups, res_cap,
                         _dt(self.k_res))
        self.B, self.Hkv, self.d, self.bits, self.group, self.residual = B, Hkv, d, bits, group, residual
        self.rotate = bool(rotate)
        self.max_groups, self.res_cap = max_groups, res_cap

    def view(self) -> CacheView:
        v = CacheView()
        v.kind = VC_CACHE_KIVI
        v.kivi = ctypes.pointer(self.c)
        return v

    def record_view(self) -> torch.Tensor:
        return self.records.view(self.B, self.Hkv, max(self.max_groups, 1), self.rec_bytes)


def dense_view(k: torch.Tensor, v: torch.Tensor, seq_len: torch.Tensor, max_len: int) -> CacheView:
    B, Hkv, Ls, d = k.shape
    cv = CacheView()
    cv.kind = VC_CACHE_DENSE
    cv.k, cv.v, cv.dt = k.data_ptr(), v.data_ptr(), _dt(k)
    cv.seq_len = seq_len.data_ptr()
    cv.B, cv.Hkv, cv.d, cv.L_stride, cv.max_len = B, Hkv, d, Ls, int(max_len)
    return cv


# ----------------------------------------------------------- entry points --

def vc_version() -> str:
    return load().vc_version().decode()


def vc_record_bytes(bits: int, d: int) -> int:
    return int(load().vc_record_bytes(bits, d))


def vc_check(stream=None):
    _check(load().vc_check(_stream(stream)), "vc_check")


def vc_workspace_init(ws: Workspace, stream=None):
    _check(load().vc_workspace_init(ws.ptr, ws.nbytes, _stream(stream)), "vc_workspace_init")


def vc_wait_probe(ws: Workspace, stream=None):
    _check(load().vc_wait_probe(ws.ptr, ws.nbytes, _stream(stream)), "vc_wait_probe")


def vc_poll_status(ws: Workspace, stream=None) -> int:
    return int(load().vc_poll_status(ws.ptr, _stream(stream)))


def vc_quantize_kv(k: torch.Tensor, v: torch.Tensor, cache: QCache, L: int | None = None, stream=None):
    B, Hkv, Ls, d = k.shape
    L = Ls if L is None else int(L)
    assert k.is_contiguous() and v.is_contiguous() and v.shape == k.shape
    _check(load().vc_quantize_kv(k.data_ptr(), v.data_ptr(), _dt(k), B, Hkv, L, Ls, d,
                                 ctypes.byref(cache.c), _stream(stream)), "vc_quantize_kv")


def vc_qcache_append(cache: QCache, k_new: torch.Tensor, v_new: torch.Tensor, n_new: torch.Tensor,
                     requantize: bool = True, stream=None):
    assert k_new.is_contiguous() and v_new.is_contiguous() and n_new.dtype == torch.int32
    max_new = k_new.shape[2]
    _check(load().vc_qcache_append(ctypes.byref(cache.c), k_new.data_ptr(), v_new.data_ptr(),
                                   n_new.data_ptr(), max_new, int(bool(requantize)), _stream(stream)),
           "vc_qcache_append")


def vc_qcache_commit(cache: QCache, k_blk: torch.Tensor, v_blk: torch.Tensor, round_len: torch.Tensor,
                     n_acc: torch.Tensor, stream=None):
    assert k_blk.is_contiguous() and v_blk.is_contiguous()
    assert round_len.dtype == torch.int32 and n_acc.dtype == torch.int32
    _check(load().vc_qcache_commit(ctypes.byref(cache.c), k_blk.data_ptr(), v_blk.data_ptr(),
                                   round_len.data_ptr(), n_acc.data_ptr(), k_blk.shape[2], _stream(stream)),
           "vc_qcache_commit")


def vc_drop_kept_count(L: int, keep_top: int, keep_recent: int) -> int:
    return int(load().vc_drop_kept_count(L, DropCfg(keep_top, keep_recent)))


def vc_drop_tokens_workspace_bytes(B, H, L) -> int:
    return int(load().vc_drop_tokens_workspace_bytes(B, H, L))


def vc_drop_tokens(scores, k, v, keep_top: int, keep_recent: int, kept_idx, k_out, v_out, ws: Workspace,
                   stream=None):
    B, H, L, d = k.shape
    assert scores.dtype == torch.float32 and scores.is_contiguous()
    _check(load().vc_drop_tokens(scores.data_ptr(), k.data_ptr(), v.data_ptr(), _dt(k), B, H, L, d,
                                 DropCfg(keep_top, keep_recent), kept_idx.data_ptr(), k_out.data_ptr(),
                                 v_out.data_ptr(), ws.ptr, ws.nbytes, _stream(stream)), "vc_drop_tokens")


def vc_draft_attn_workspace_bytes(view: CacheView, Hq: int) -> int:
    return int(load().vc_draft_attn_workspace_bytes(ctypes.byref(view), Hq))


def vc_draft_attn(q: torch.Tensor, view: CacheView, sm_scale: float, out: torch.Tensor, ws: Workspace,
                  stream=None):
    B, Hq, d = q.shape
    assert q.is_contiguous() and out.is_contiguous()
    _check(load().vc_draft_attn(q.data_ptr(), _dt(q), ctypes.byref(view), Hq, sm_scale, out.data_ptr(), ws.ptr,
                                ws.nbytes, _stream(stream)), "vc_draft_attn")


def vc_draft_attn_h2o_workspace_bytes(view: CacheView, Hq: int) -> int:
    return int(load().vc_draft_attn_h2o_workspace_bytes(ctypes.byref(view), Hq))


def vc_draft_attn_h2o(q: torch.Tensor, view: CacheView, sm_scale: float, out: torch.Tensor, scores: torch.Tensor,
                      ws: Workspace, kept_idx: torch.Tensor | None = None, stream=None):
    """scores: fp32 [B][Hkv][S] (S = original positions); kept_idx: int32
    [B][Hkv][n_keep] mapping the view's rows to positions, or None."""
    B, Hq, d = q.shape
    assert q.is_contiguous() and out.is_contiguous() and scores.dtype == torch.float32 and scores.is_contiguous()
    ks = kept_idx.shape[-1] if kept_idx is not None else 0
    _check(load().vc_draft_attn_h2o(q.data_ptr(), _dt(q), ctypes.byref(view), Hq, sm_scale, out.data_ptr(),
                                    scores.data_ptr(), scores.shape[-1], _ptr(kept_idx), ks, ws.ptr, ws.nbytes,
                                    _stream(stream)), "vc_draft_attn_h2o")


def vc_verify_attn_workspace_bytes(dtype, B, Dq, Hq, Hkv, d, max_ctx) -> int:
    dt = VC_BF16 if dtype == torch.bfloat16 else VC_F32
    return int(load().vc_verify_attn_workspace_bytes(dt, B, Dq, Hq, Hkv, d, max_ctx))


def vc_verify_attn(q, k, v, ctx_len, max_ctx: int, sm_scale: float, out, ws: Workspace, stream=None):
    B, Dq, Hq, d = q.shape
    _, Hkv, Ls, _ = k.shape
    assert q.is_contiguous() and k.is_contiguous() and v.is_contiguous() and ctx_len.dtype == torch.int32
    _check(load().vc_verify_attn(q.data_ptr(), k.data_ptr(), v.data_ptr(), _dt(q), ctx_len.data_ptr(), B, Dq, Hq,
                                 Hkv, d, Ls, int(max_ctx), sm_scale, out.data_ptr(), ws.ptr, ws.nbytes,
                                 _stream(stream)), "vc_verify_attn")


def vc_verify_attn_h2o_workspace_bytes(B, Dq, Hq, Hkv, d, max_ctx) -> int:
    return int(load().vc_verify_attn_h2o_workspace_bytes(B, Dq, Hq, Hkv, d, max_ctx))


def vc_verify_attn_h2o(q, k, v, ctx_len, max_ctx: int, sm_scale: float, out, scores, ws: Workspace, stream=None):
    """vc_verify_attn plus H2O accumulation into scores fp32 [B][Hkv][S]
    (S >= max_ctx + Dq: one entry per key position)."""
    B, Dq, Hq, d = q.shape
    _, Hkv, Ls, _ = k.shape
    assert q.is_contiguous() and k.is_contiguous() and v.is_contiguous() and ctx_len.dtype == torch.int32
    assert scores.dtype == torch.float32 and scores.is_contiguous() and scores.shape[:2] == (B, Hkv)
    _check(load().vc_verify_attn_h2o(q.data_ptr(), k.data_ptr(), v.data_ptr(), ctx_len.data_ptr(), B, Dq, Hq, Hkv,
                                     d, Ls, int(max_ctx), sm_scale, out.data_ptr(), scores.data_ptr(),
                                     scores.shape[2], ws.ptr, ws.nbytes, _stream(stream)), "vc_verify_attn_h2o")


def vc_accept_workspace_bytes(B, D, V) -> int:
    return int(load().vc_accept_workspace_bytes(B, D, V))


def vc_accept(logits, drafts, n_acc, next_tok, ws: Workspace, stream=None):
    B, D1, V = logits.shape
    assert logits.is_contiguous()
    dp = drafts.data_ptr() if drafts is not None and drafts.numel() else None
    _check(load().vc_accept(logits.data_ptr(), _dt(logits), dp, B, D1 - 1, V, n_acc.data_ptr(),
                            next_tok.data_ptr(), ws.ptr, ws.nbytes, _stream(stream)), "vc_accept")


def vc_accept_noalloc(logits, drafts, n_acc, next_tok, stream=None):
    """vc_accept without a workspace: the library's static device buffer is
    used instead (for callers that cannot allocate; see include/vc.h)."""
    B, D1, V = logits.shape
    assert logits.is_contiguous()
    dp = drafts.data_ptr() if drafts is not None and drafts.numel() else None
    _check(load().vc_accept_noalloc(logits.data_ptr(), _dt(logits), dp, B, D1 - 1, V, n_acc.data_ptr(),
                                    next_tok.data_ptr(), _stream(stream)), "vc_accept_noalloc")


def vc_swap_in(dst: torch.Tensor, src_pinned: torch.Tensor, nbytes: int | None = None, stream=None,
               done_event: torch.cuda.Event | None = None):
    n = dst.numel() * dst.element_size() if nbytes is None else int(nbytes)
    ev = None
    if done_event is not None:
        if not done_event.cuda_event:          # torch creates the event lazily
            done_event.record(torch.cuda.current_stream() if stream is None else stream)
        ev = done_event.cuda_event
    _check(load().vc_swap_in(dst.data_ptr(), src_pinned.data_ptr(), n, _stream(stream), ev), "vc_swap_in")


def vc_swap_in_rows(dst: torch.Tensor, src_pinned: torch.Tensor, rows: int, stream=None,
                    done_event: torch.cuda.Event | None = None):
    """The first `rows` rows of every block of a [..][pitch_rows][row] tensor
    pair (the last two dimensions are rows and the row's elements): one 2-D
    copy from pinned host memory (include/vc.h, vc_swap_in_rows)."""
    assert dst.shape == src_pinned.shape and dst.is_contiguous() and src_pinned.is_contiguous()
    pitch_rows = dst.shape[-2]
    row_bytes = dst.shape[-1] * dst.element_size()
    blocks = dst.numel() // (dst.shape[-1] * pitch_rows)
    ev = None
    if done_event is not None:
        if not done_event.cuda_event:          # torch creates the event lazily
            done_event.record(torch.cuda.current_stream() if stream is None else stream)
        ev = done_event.cuda_event
    _check(load().vc_swap_in_rows(dst.data_ptr(), src_pinned.data_ptr(), row_bytes, min(int(rows), pitch_rows),
                                  pitch_rows, blocks, _stream(stream), ev), "vc_swap_in_rows")


# ---------------------------------------------------------------- decoder --

def vc_gemm_workspace_bytes(dtype, M, N, K) -> int:
    dt = VC_BF16 if dtype == torch.bfloat16 else VC_F32
    return int(load().vc_gemm_workspace_bytes(dt, M, N, K))


def vc_gemm_splits(dtype, N, K, decode_plan: bool = False) -> int:
    dt = VC_BF16 if dtype == torch.bfloat16 else VC_F32
    return int(load().vc_gemm_splits(dt, N, K, int(bool(decode_plan))))


def vc_gemm(x, w, out, resid=None, ws: Workspace | None = None, stream=None, decode_plan: bool = False):
    M, K = x.shape
    K2, N = w.shape
    assert K == K2 and out.shape == (M, N) and x.is_contiguous() and w.is_contiguous() and out.is_contiguous()
    _check(load().vc_gemm_ex(x.data_ptr(), w.data_ptr(), _ptr(resid), out.data_ptr(), _dt(x), M, N, K,
                             int(bool(decode_plan)), ws.ptr if ws is not None else None,
                             ws.nbytes if ws is not None else 0, _stream(stream)), "vc_gemm")


def vc_gemm_argmax(x, w, tile_max, tile_idx, ws: Workspace | None = None, stream=None, decode_plan: bool = False):
    """Tile maxima of bf16(x W): tile_max float32 [M][N/128], tile_idx int32."""
    M, K = x.shape
    K2, N = w.shape
    assert K == K2 and x.is_contiguous() and w.is_contiguous()
    assert tile_max.shape == (M, N // 128) and tile_idx.shape == (M, N // 128)
    assert tile_max.dtype == torch.float32 and tile_idx.dtype == torch.int32
    _check(load().vc_gemm_argmax(x.data_ptr(), w.data_ptr(), _dt(x), M, N, K, int(bool(decode_plan)),
                                 tile_max.data_ptr(), tile_idx.data_ptr(), ws.ptr if ws is not None else None,
                                 ws.nbytes if ws is not None else 0, _stream(stream)), "vc_gemm_argmax")


def interleave_gate_up(wg: torch.Tensor, wu: torch.Tensor) -> torch.Tensor:
    """The decoder's gate|up weight layout (include/vc.h, vc_decoder_weights):
    [K][F] gate and up columns interleaved per 64 into [K][2F]."""
    K, F = wg.shape
    assert wu.shape == (K, F) and F % 64 == 0
    return torch.stack([wg.reshape(K, F // 64, 64), wu.reshape(K, F // 64, 64)], dim=2).reshape(K, 2 * F)


def vc_gemm_rms(x, w, out, eps: float, swiglu: bool = False, ws: Workspace | None = None, stream=None):
    """out = rmsnorm(x) W (swiglu: the SwiGLU of it, W interleaved gate|up,
    out [M][N/2]) with the normalisation in the GEMM epilogue, as the
    decoder's draft steps compute it (bf16, M <= 16)."""
    M, K = x.shape
    K2, N = w.shape
    assert K == K2 and out.shape == ((M, N // 2) if swiglu else (M, N))
    assert x.is_contiguous() and w.is_contiguous() and out.is_contiguous()
    _check(load().vc_gemm_rms(x.data_ptr(), w.data_ptr(), out.data_ptr(), _dt(x), M, N, K, float(eps),
                              int(bool(swiglu)), ws.ptr if ws is not None else None,
                              ws.nbytes if ws is not None else 0, _stream(stream)), "vc_gemm_rms")


def vc_gemm_swiglu(x, w_gate_up, act, stream=None, decode_plan: bool = False):
    """act [M][F] = silu(g) * u of the bf16-rounded gate and up products of
    x [M][K] with w_gate_up [K][2F] (interleaved layout), in the GEMM epilogue."""
    M, K = x.shape
    K2, N = w_gate_up.shape
    assert K == K2 and act.shape == (M, N // 2)
    assert x.is_contiguous() and w_gate_up.is_contiguous() and act.is_contiguous()
    _check(load().vc_gemm_swiglu(x.data_ptr(), w_gate_up.data_ptr(), act.data_ptr(), _dt(x), M, N // 2, K,
                                 int(bool(decode_plan)), _stream(stream)), "vc_gemm_swiglu")


def vc_accept_tiles(tile_max, tile_idx, drafts, n_acc, next_tok, stream=None):
    """tile_max/tile_idx: [B][D+1][n_tiles]; same outputs as vc_accept."""
    B, D1, nt = tile_max.shape
    assert tile_max.is_contiguous() and tile_idx.is_contiguous()
    dp = drafts.data_ptr() if drafts is not None and drafts.numel() else None
    _check(load().vc_accept_tiles(tile_max.data_ptr(), tile_idx.data_ptr(), nt, dp, B, D1 - 1, n_acc.data_ptr(),
                                  next_tok.data_ptr(), _stream(stream)), "vc_accept_tiles")


class Decoder:
    """A vc_decoder handle plus the device weights it points to (kept alive
    here).  `weights` is a dict of tensors stored [in][out]: embed, lm_head
    and per layer wq, wk, wv, wo, wg, wu, wd; the q|k|v and gate|up column
    blocks are laid side by side once here, as the C ABI expects."""

    def __init__(self, cfg, weights: dict, dtype=torch.bfloat16, device="cuda"):
        def dev(t):
            return t.to(device=device, dtype=dtype).contiguous()
        self.cfg, self.dtype = cfg, dtype
        self.embed = dev(weights["embed"])
        self.lm_head = dev(weights["lm_head"])
        self.wqkv, self.wo, self.wgu, self.wd = [], [], [], []
        for lw in weights["layers"]:
            self.wqkv.append(torch.cat([dev(lw["wq"]), dev(lw["wk"]), dev(lw["wv"])], dim=1).contiguous())
            self.wo.append(dev(lw["wo"]))
            self.wgu.append(interleave_gate_up(dev(lw["wg"]), dev(lw["wu"])).contiguous())
            self.wd.append(dev(lw["wd"]))
        self._init_handle()

    @classmethod
    def from_packed(cls, cfg, embed, lm_head, wqkv, wo, wgu, wd, dtype=torch.bfloat16):
        """Weights already laid out as the C ABI wants them (device tensors)."""
        self = cls.__new__(cls)
        self.cfg, self.dtype = cfg, dtype
        self.embed, self.lm_head = embed, lm_head
        self.wqkv, self.wo, self.wgu, self.wd = list(wqkv), list(wo), list(wgu), list(wd)
        self._init_handle()
        return self

    def _init_handle(self):
        cfg = self.cfg
        n = cfg.n_layers
        arr = ctypes.c_void_p * n
        self._arrs = [arr(*[t.data_ptr() for t in ts]) for ts in (self.wqkv, self.wo, self.wgu, self.wd)]
        w = DecoderWeights(self.embed.data_ptr(), self.lm_head.data_ptr(), *self._arrs)
        c = DecoderCfg(cfg.n_layers, cfg.d_model, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.d_ff, cfg.vocab,
                       cfg.norm_eps, cfg.rope_theta, VC_BF16 if self.dtype == torch.bfloat16 else VC_F32)
        h = c_void_p()
        _check(load().vc_decoder_create(ctypes.byref(c), ctypes.byref(w), ctypes.byref(h)), "vc_decoder_create")
        self.handle = h

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and h.value and _lib is not None:
            _lib.vc_decoder_destroy(h)
            self.handle = None

    def workspace_bytes(self, B: int, max_rows: int, max_ctx: int, draft_cache: "QCache | None" = None) -> int:
        dc = ctypes.byref(draft_cache.c) if draft_cache is not None else None
        return int(load().vc_decoder_workspace_bytes(self.handle, B, max_rows, max_ctx, dc))


def vc_decoder_forward(dec: Decoder, first_tok, tokens, tok_stride: int, B: int, Dq: int, ctx_len, max_ctx: int,
                       k_cache, v_cache, logits, ws: Workspace, k_blk=None, v_blk=None, last_only=False,
                       stream=None):
    L_stride = k_cache.shape[3]
    _check(load().vc_decoder_forward(dec.handle, _ptr(first_tok), _ptr(tokens), int(tok_stride), B, Dq,
                                     ctx_len.data_ptr(), int(max_ctx), k_cache.data_ptr(), v_cache.data_ptr(),
                                     L_stride, _ptr(k_blk), _ptr(v_blk), int(bool(last_only)), logits.data_ptr(),
                                     ws.ptr, ws.nbytes, _stream(stream)), "vc_decoder_forward")


def vc_decoder_verify(dec: Decoder, first_tok, drafts, D: int, B: int, ctx_len, max_ctx: int, k_cache, v_cache,
                      n_acc, next_tok, ws: Workspace, k_blk=None, v_blk=None, stream=None):
    """Verify pass plus greedy acceptance without logits (vc_decoder_verify)."""
    L_stride = k_cache.shape[3]
    _check(load().vc_decoder_verify(dec.handle, first_tok.data_ptr(), _ptr(drafts), int(D), B, ctx_len.data_ptr(),
                                    int(max_ctx), k_cache.data_ptr(), v_cache.data_ptr(), L_stride, _ptr(k_blk),
                                    _ptr(v_blk), n_acc.data_ptr(), next_tok.data_ptr(), ws.ptr, ws.nbytes,
                                    _stream(stream)), "vc_decoder_verify")


def qcache_array(caches: list):
    """The host array of vc_qcache structs that vc_decoder_draft_step takes
    (one per layer; the structs are copied, the storage stays in `caches`)."""
    return (QCacheC * len(caches))(*[c.c for c in caches])


def vc_decoder_draft_step(dec: Decoder, tok, caches_arr, logits, next_tok, ws: Workspace, drafts_out=None,
                          drafts_stride: int = 1, stream=None):
    """caches_arr: qcache_array(caches) (built once per set of caches); logits
    None runs the LM head with the argmax epilogue (no logits written)."""
    _check(load().vc_decoder_draft_step(dec.handle, tok.data_ptr(), tok.shape[0], caches_arr, _ptr(logits),
                                        next_tok.data_ptr(), _ptr(drafts_out), int(drafts_stride), ws.ptr,
                                        ws.nbytes, _stream(stream)), "vc_decoder_draft_step")


def vc_kv_writeback(k_blk, v_blk, n_acc, ctx_len, k_host, v_host, stream=None):
    nl, B, Hkv, Dq, d = k_blk.shape
    L_stride = k_host.shape[3]
    _check(load().vc_kv_writeback(k_blk.data_ptr(), v_blk.data_ptr(), _dt(k_blk), nl, B, Hkv, Dq, d,
                                  n_acc.data_ptr(), ctx_len.data_ptr(), k_host.data_ptr(), v_host.data_ptr(),
                                  L_stride, _stream(stream)), "vc_kv_writeback")


def vc_decoder_set_layer_events(dec: Decoder, events: list | None):
    """Per-layer arrival events of a full cache being copied in: the decoder's
    forward and verify wait on events[l] before touching layer l (include/vc.h,
    vc_decoder_set_layer_events).  events: one torch.cuda.Event per layer,
    recorded by the caller on the copying stream; None clears them."""
    if not events:
        _check(load().vc_decoder_set_layer_events(dec.handle, None, 0), "vc_decoder_set_layer_events")
        return
    for e in events:                                 # torch creates events lazily
        if not e.cuda_event:
            e.record()
    arr = (c_void_p * len(events))(*[e.cuda_event for e in events])
    _check(load().vc_decoder_set_layer_events(dec.handle, arr, len(events)), "vc_decoder_set_layer_events")


class DecoderTrace:
    """Event pairs the decoder records around its GEMMs and attention calls
    (vc_decoder_set_trace); capacity = operations to record."""

    def __init__(self, dec: Decoder, capacity: int, kinds=TRACE_KINDS):
        self.dec, self.capacity = dec, capacity
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(2 * capacity)]
        for e in self.events:                       # torch creates events lazily
            e.record()
        torch.cuda.synchronize()
        self._ev_arr = (c_void_p * (2 * capacity))(*[e.cuda_event for e in self.events])
        self._kinds = (c_int32 * capacity)()
        self.mask = sum(1 << TRACE_KINDS.index(k) for k in kinds)

    def start(self):
        _check(load().vc_decoder_set_trace(self.dec.handle, self._ev_arr, self._kinds, self.capacity, self.mask),
               "vc_decoder_set_trace")

    def stop(self) -> list[tuple[str, float]]:
        """Turn tracing off; returns (kind, milliseconds) per recorded operation
        (synchronizes)."""
        self.n = int(load().vc_decoder_trace_count(self.dec.handle))
        _check(load().vc_decoder_set_trace(self.dec.handle, None, None, 0, 0), "vc_decoder_set_trace")
        torch.cuda.synchronize()
        return self.times()

    def times(self, first: int = 0, count: int | None = None) -> list[tuple[str, float]]:
        """(kind, milliseconds) of traced operations first .. first + count - 1
        as last recorded (for a trace captured into a graph: the last replay)."""
        n = self.n if count is None else count
        return [(TRACE_KINDS[self._kinds[k]], self.events[2 * k].elapsed_time(self.events[2 * k + 1]))
                for k in range(first, first + n)]


def vc_kv_packed_row_bytes(d: int) -> int:
    return int(load().vc_kv_packed_row_bytes(d))


def vc_kv_pack(src: torch.Tensor, dst: torch.Tensor, n_over: torch.Tensor | None = None, stream=None):
    """src bf16 [..., d] (rows = everything before d) -> dst uint8 [..., 16 + 3d/2]
    (device, or pinned host mapped into the device); n_over: int32 device
    counter of rows that cannot be packed (added to)."""
    d = src.shape[-1]
    rows = src.numel() // d if d else 0
    assert src.dtype == torch.bfloat16 and src.is_contiguous() and dst.dtype == torch.uint8 and dst.is_contiguous()
    assert dst.numel() == rows * vc_kv_packed_row_bytes(d)
    _check(load().vc_kv_pack(src.data_ptr(), dst.data_ptr(), rows, d, _ptr(n_over), _stream(stream)), "vc_kv_pack")


def vc_kv_unpack(src: torch.Tensor, dst: torch.Tensor, stream=None):
    """src uint8 [..., 16 + 3d/2] (device) -> dst bf16 [..., d]."""
    d = dst.shape[-1]
    rows = dst.numel() // d if d else 0
    assert dst.dtype == torch.bfloat16 and dst.is_contiguous() and src.dtype == torch.uint8 and src.is_contiguous()
    assert src.numel() == rows * vc_kv_packed_row_bytes(d)
    _check(load().vc_kv_unpack(src.data_ptr(), dst.data_ptr(), rows, d, _stream(stream)), "vc_kv_unpack")


def vc_kv_writeback_packed(k_blk, v_blk, n_acc, ctx_len, k_host_packed, v_host_packed, n_over=None, stream=None):
    """k_blk/v_blk bf16 [n_layers][B][Hkv][Dq][d] (device); the host copies
    pinned uint8 [n_layers][B][Hkv][L_stride][16 + 3d/2]."""
    nl, B, hkv, dq, d = k_blk.shape
    L_stride = k_host_packed.shape[3]
    assert k_host_packed.shape == (nl, B, hkv, L_stride, vc_kv_packed_row_bytes(d)) == v_host_packed.shape
    _check(load().vc_kv_writeback_packed(k_blk.data_ptr(), v_blk.data_ptr(), nl, B, hkv, dq, d, n_acc.data_ptr(),
                                         ctx_len.data_ptr(), k_host_packed.data_ptr(), v_host_packed.data_ptr(),
                                         L_stride, _ptr(n_over), _stream(stream)), "vc_kv_writeback_packed")


def vc_swap_in_paced(dst: torch.Tensor, src_pinned: torch.Tensor, gbps: float, pace_ws: torch.Tensor,
                     chunk_bytes: int = 64 << 20, stream=None, done_event: torch.cuda.Event | None = None):
    """vc_swap_in at an emulated source rate of `gbps` GB/s (see include/vc.h);
    pace_ws: a 16-byte device tensor owned by the caller."""
    n = dst.numel() * dst.element_size()
    ev = None
    if done_event is not None:
        if not done_event.cuda_event:
            done_event.record(torch.cuda.current_stream() if stream is None else stream)
        ev = done_event.cuda_event
    _check(load().vc_swap_in_paced(dst.data_ptr(), src_pinned.data_ptr(), n, float(gbps), int(chunk_bytes),
                                   pace_ws.data_ptr(), _stream(stream), ev), "vc_swap_in_paced")
