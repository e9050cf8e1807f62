"""ctypes binding of the attention C ABI (``include/attn.h``).

Argument marshalling only: every step of the computation runs in the CUDA
library ``libattn_sm103.so``.  PyTorch supplies device memory and the stream.
Loading fails loudly (RuntimeError) when the library is missing; there is no
fallback implementation.
"""
from __future__ import annotations

import contextlib
import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libattn_sm103.so")

ATTN_PARAMS_VERSION = 6

LAYOUTS = {"3HD": 0, "HD_2HD": 1, "HD_HD_HD": 2}
FORMATS = {"BSHD": 0, "THD_SEGMENTS": 1, "THD_CU_SEQLENS": 2}
MASKS = {"NONE": 0, "CAUSAL": 1, "PADDING": 2, "PADDING_CAUSAL": 3}
DQ_MODES = {"atomic": 0, "deterministic": 1}
DTYPES = {"bf16": 0, "fp16": 1, "fp8_e4m3": 2}
STATUS = {0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED",
          3: "ATTN_ERR_SHAPE_MISMATCH", 4: "ATTN_ERR_WORKSPACE_TOO_SMALL", 5: "ATTN_ERR_CUDA",
          6: "ATTN_ERR_DEVICE_TIMEOUT", 7: "ATTN_ERR_DEVICE_BOUNDS"}
BUILD_DEVICE_CHECKS = 1
EXPORTED = ("attn_abi_version", "attn_status_string", "attn_fwd_workspace_size",
            "attn_bwd_workspace_size", "attn_resolve_layout", "attn_fwd", "attn_bwd",
            "attn_read_status", "attn_set_trace_events", "attn_event_create",
            "attn_event_destroy", "attn_event_elapsed_ms", "attn_fwd_noalloc",
            "attn_build_flags")
FWD_NOALLOC_SCRATCH_BYTES = 4 << 20
TRACE_SLOTS = ("meta", "fwd", "bwd_pre", "dkdv", "dq", "dbias")

c_i32, c_i64, c_f32, c_vp, c_sz = (ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                                   ctypes.c_void_p, ctypes.c_size_t)


class attn_params_t(ctypes.Structure):
    _fields_ = [
        ("struct_version", c_i32), ("fmt", c_i32), ("layout", c_i32), ("mask", c_i32),
        ("dq_mode", c_i32),
        ("B", c_i32), ("Sq", c_i32), ("Skv", c_i32), ("Hq", c_i32), ("Hkv", c_i32),
        ("d_qk", c_i32), ("d_v", c_i32),
        ("scale", c_f32),
        ("q", c_vp), ("k", c_vp), ("v", c_vp),
        ("q_seg_ids", c_vp), ("q_seg_pos", c_vp), ("kv_seg_ids", c_vp), ("kv_seg_pos", c_vp),
        ("q_ids_dims", c_i64 * 2), ("q_pos_dims", c_i64 * 2), ("kv_ids_dims", c_i64 * 2),
        ("kv_pos_dims", c_i64 * 2),
        ("cu_seqlens_q", c_vp), ("cu_seqlens_kv", c_vp), ("num_segments", c_i32),
        ("bias", c_vp), ("bias_b", c_i32), ("bias_h", c_i32),
        ("force_general_path", c_i32),
        ("metadata_from_forward", c_i32),
        ("max_logit", c_vp),
        ("sink", c_vp), ("dsink", c_vp),
        ("band", c_i32), ("window_left", c_i32), ("window_right", c_i32),
        ("bottom_right", c_i32),
        ("dtype", c_i32),
        ("test_wait_timeout", c_i32),
        ("descale_q", c_f32), ("descale_k", c_f32), ("descale_v", c_f32),
    ]


class attn_stats_t(ctypes.Structure):
    _fields_ = [("status", c_i32), ("path", c_i32), ("reason", c_i32), ("dq_mode", c_i32),
                ("tile_pairs", c_i64), ("wait_site", c_i32), ("reserved", c_i32)]


class attn_resolved_t(ctypes.Structure):
    _fields_ = [("q", c_vp), ("k", c_vp), ("v", c_vp), ("q_token_stride", c_i64),
                ("k_token_stride", c_i64), ("v_token_stride", c_i64), ("dq", c_vp), ("dk", c_vp),
                ("dv", c_vp)]


_lib = None


def load_library(path: str = LIB_PATH):
    """Load the CUDA library (built by ``bwd_tcgen05_tma_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA attention library not built: {path} is missing "
                           "(run bwd_tcgen05_tma_gb300.build.build())")
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER(attn_params_t)
    lib.attn_abi_version.restype = c_i32
    lib.attn_build_flags.restype = c_i32
    lib.attn_status_string.restype = ctypes.c_char_p
    lib.attn_status_string.argtypes = [c_i32]
    lib.attn_fwd_workspace_size.restype = c_sz
    lib.attn_fwd_workspace_size.argtypes = [P]
    lib.attn_bwd_workspace_size.restype = c_sz
    lib.attn_bwd_workspace_size.argtypes = [P]
    lib.attn_resolve_layout.restype = c_i32
    lib.attn_resolve_layout.argtypes = [P, c_vp, c_vp, c_vp, ctypes.POINTER(attn_resolved_t)]
    lib.attn_fwd.restype = c_i32
    lib.attn_fwd.argtypes = [P, c_vp, c_vp, c_vp, c_sz, c_vp]
    lib.attn_bwd.restype = c_i32
    lib.attn_bwd.argtypes = [P, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_sz, c_vp]
    lib.attn_read_status.restype = c_i32
    lib.attn_read_status.argtypes = [c_vp, c_vp, ctypes.POINTER(attn_stats_t)]
    lib.attn_set_trace_events.restype = c_i32
    lib.attn_set_trace_events.argtypes = [ctypes.POINTER(c_vp)]
    lib.attn_fwd_noalloc.restype = c_i32
    lib.attn_fwd_noalloc.argtypes = [P, c_vp, c_vp, c_vp]
    lib.attn_event_create.restype = c_i32
    lib.attn_event_create.argtypes = [ctypes.POINTER(c_vp)]
    lib.attn_event_destroy.restype = c_i32
    lib.attn_event_destroy.argtypes = [c_vp]
    lib.attn_event_elapsed_ms.restype = c_i32
    lib.attn_event_elapsed_ms.argtypes = [c_vp, c_vp, ctypes.POINTER(ctypes.c_float)]
    if lib.attn_abi_version() != ATTN_PARAMS_VERSION:
        raise RuntimeError("attention library ABI version mismatch")
    _lib = lib
    return lib


@contextlib.contextmanager
def library_scope(path: str):
    """Route every call made inside the block to the library at ``path`` (for
    example the checking build, ``build.build(debug=True)``); the library
    loaded before is restored afterwards."""
    global _lib
    prev = _lib
    _lib = None
    try:
        yield load_library(path)
    finally:
        _lib = prev


class AttnError(RuntimeError):
    def __init__(self, code, what):
        self.code = code
        name = STATUS.get(code, str(code))
        msg = load_library().attn_status_string(code).decode()
        super().__init__(f"{what}: {name} ({msg})")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch

        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(getattr(stream, "cuda_stream", stream))


def make_params(*, layout, fmt, mask, B, Sq, Skv, Hq, Hkv, d_qk, d_v, scale, q, k=None, v=None,
                q_seg_ids=None, q_seg_pos=None, kv_seg_ids=None, kv_seg_pos=None,
                cu_seqlens_q=None, cu_seqlens_kv=None, bias=None, dq_mode="deterministic",
                force_general_path=False, metadata_from_forward=False, max_logit=None,
                sink=None, dsink=None, window=None, bottom_right=False, dtype="bf16",
                descale=(1.0, 1.0, 1.0)):
    """Fill an ``attn_params_t`` from tensors (any object with data_ptr/shape).
    max_logit: optional fp32 [B, Hq] tensor the forward fills; sink: optional
    fp32 [Hq] sink logits; dsink: optional fp32 [Hq] tensor the backward fills
    with their gradient; window: optional (left, right) band, None for an
    unbounded side; bottom_right: align positions by Skv - Sq; dtype: "bf16",
    "fp16" or "fp8_e4m3" (forward only: Q / K / V as E4M3 codes, O in bf16);
    descale: the (q, k, v) factors the E4M3 codes stand scaled by (see attn.h)."""
    p = attn_params_t()
    p.struct_version = ATTN_PARAMS_VERSION
    p.fmt = FORMATS[fmt]
    p.layout = LAYOUTS[layout]
    p.mask = MASKS[mask]
    p.dq_mode = DQ_MODES[dq_mode]
    p.B, p.Sq, p.Skv, p.Hq, p.Hkv, p.d_qk, p.d_v = B, Sq, Skv, Hq, Hkv, d_qk, d_v
    p.scale = float(scale)
    p.q, p.k, p.v = _ptr(q), _ptr(k), _ptr(v)
    for name, t in (("q_seg_ids", q_seg_ids), ("q_seg_pos", q_seg_pos), ("kv_seg_ids", kv_seg_ids),
                    ("kv_seg_pos", kv_seg_pos)):
        setattr(p, name, _ptr(t))
        if t is not None:
            dims = tuple(t.shape)
            if len(dims) == 1:
                dims = (1,) + dims
            key = {"q_seg_ids": "q_ids_dims", "q_seg_pos": "q_pos_dims",
                   "kv_seg_ids": "kv_ids_dims", "kv_seg_pos": "kv_pos_dims"}[name]
            arr = getattr(p, key)
            arr[0] = int(dims[-2]) if len(dims) >= 2 else 1
            arr[1] = int(dims[-1])
            if len(dims) > 2:  # extra leading dims: a mismatch the library reports
                arr[0] = -1
    p.cu_seqlens_q, p.cu_seqlens_kv = _ptr(cu_seqlens_q), _ptr(cu_seqlens_kv)
    p.num_segments = 0 if cu_seqlens_q is None else int(cu_seqlens_q.shape[0]) - 1
    p.bias = _ptr(bias)
    if bias is not None:
        p.bias_b, p.bias_h = int(bias.shape[0]), int(bias.shape[1])
    p.force_general_path = 1 if force_general_path else 0
    p.metadata_from_forward = 1 if metadata_from_forward else 0
    p.max_logit = _ptr(max_logit)
    p.sink = _ptr(sink)
    p.dsink = _ptr(dsink)
    if window is not None:
        left, right = window
        p.band = 1
        p.window_left = -1 if left is None else int(left)
        p.window_right = -1 if right is None else int(right)
    p.bottom_right = 1 if bottom_right else 0
    p.dtype = DTYPES[dtype]
    p.descale_q, p.descale_k, p.descale_v = (float(x) for x in descale)
    return p


def attn_fwd_workspace_size(p):
    return int(load_library().attn_fwd_workspace_size(ctypes.byref(p)))


def attn_bwd_workspace_size(p):
    return int(load_library().attn_bwd_workspace_size(ctypes.byref(p)))


def attn_resolve_layout(p, dq=None, dk=None, dv=None):
    r = attn_resolved_t()
    s = load_library().attn_resolve_layout(ctypes.byref(p), dq, dk, dv, ctypes.byref(r))
    if s != 0:
        raise AttnError(s, "attn_resolve_layout")
    return r


def attn_fwd(p, o, lse, ws, stream=None):
    """Enqueue the forward on `stream` (default: torch's current stream)."""
    s = load_library().attn_fwd(ctypes.byref(p), _ptr(o), _ptr(lse), _ptr(ws),
                                ws.numel() * ws.element_size(), _stream(stream))
    if s != 0:
        raise AttnError(s, "attn_fwd")


def attn_fwd_noalloc(p, o, lse, stream=None):
    """Forward without a workspace: the library's fixed device scratch array is
    used instead (no allocation).  For callers that cannot allocate device
    memory at run time.  Overlapping calls on the GPU race on that array."""
    s = load_library().attn_fwd_noalloc(ctypes.byref(p), _ptr(o), _ptr(lse), _stream(stream))
    if s != 0:
        raise AttnError(s, "attn_fwd_noalloc")


def attn_bwd(p, o, d_o, lse, dq, dk, dv, dbias, ws, stream=None):
    """Enqueue the backward on `stream` (default: torch's current stream)."""
    s = load_library().attn_bwd(ctypes.byref(p), _ptr(o), _ptr(d_o), _ptr(lse), _ptr(dq), _ptr(dk),
                                _ptr(dv), _ptr(dbias), _ptr(ws), ws.numel() * ws.element_size(),
                                _stream(stream))
    if s != 0:
        raise AttnError(s, "attn_bwd")


def attn_read_status(ws, stream=None):
    """Synchronise and return (status, attn_stats_t) of the last call on `ws`."""
    st = attn_stats_t()
    s = load_library().attn_read_status(_ptr(ws), _stream(stream), ctypes.byref(st))
    return s, st


class Event:
    """A CUDA timing event owned by this object (created through the library)."""

    def __init__(self):
        h = c_vp()
        s = load_library().attn_event_create(ctypes.byref(h))
        if s != 0:
            raise AttnError(s, "attn_event_create")
        self.handle = h.value

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.attn_event_destroy(self.handle)
            self.handle = None


def attn_event_elapsed_ms(start, end):
    """Milliseconds between two recorded events, or None if either is unrecorded."""
    ms = ctypes.c_float()
    s = load_library().attn_event_elapsed_ms(start.handle, end.handle, ctypes.byref(ms))
    return float(ms.value) if s == 0 else None


def attn_set_trace_events(events):
    """events: None, or a sequence of 2 * len(TRACE_SLOTS) Event objects (or None)
    as (start, end) per slot.  The caller keeps the events alive."""
    lib = load_library()
    if events is None:
        return lib.attn_set_trace_events(None)
    arr = (c_vp * (2 * len(TRACE_SLOTS)))()
    for i, e in enumerate(events):
        arr[i] = None if e is None else c_vp(e.handle)
    s = lib.attn_set_trace_events(arr)
    if s != 0:
        raise AttnError(s, "attn_set_trace_events")
