"""Host-side C ABI checks (no GPU needed): the library builds and loads, every
symbol the header declares is exported, and validation, layout resolution and
workspace sizing behave as documented.  Only host-only entry points are
called; pointers are fake addresses that the library never dereferences."""
import ctypes
import os
import re

import pytest

from bwd_tcgen05_tma_gb300 import attn as A

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = 0x10000000


@pytest.fixture(scope="module")
def lib():
    from bwd_tcgen05_tma_gb300 import build

    build.build()
    return A.load_library()


def header_functions():
    src = open(os.path.join(ROOT, "include", "attn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = header_functions()
    assert set(names) == set(A.EXPORTED)
    for n in names:
        assert hasattr(lib, n), n


def params(**kw):
    d = dict(layout="HD_HD_HD", fmt="BSHD", mask="CAUSAL", B=2, Sq=256, Skv=256, Hq=8, Hkv=2,
             d_qk=128, d_v=128, scale=0.088)
    d.update(kw)
    p = A.attn_params_t()
    p.struct_version = A.ATTN_PARAMS_VERSION
    p.fmt, p.layout, p.mask = A.FORMATS[d["fmt"]], A.LAYOUTS[d["layout"]], A.MASKS[d["mask"]]
    p.dq_mode = 1
    p.B, p.Sq, p.Skv, p.Hq, p.Hkv, p.d_qk, p.d_v = (d[k] for k in
                                                     ("B", "Sq", "Skv", "Hq", "Hkv", "d_qk", "d_v"))
    p.scale = d["scale"]
    p.q, p.k, p.v = FAKE, FAKE + (1 << 24), FAKE + (2 << 24)
    return p


def test_workspace_sizes(lib):
    p = params()
    f, b = A.attn_fwd_workspace_size(p), A.attn_bwd_workspace_size(p)
    assert 0 < f < b and f % 256 == 0 and b % 256 == 0
    p.dq_mode = 0  # atomic: fp32 dQ accumulator in the workspace
    assert A.attn_bwd_workspace_size(p) >= b + 2 * 256 * 8 * 128 * 4
    bad = params(d_qk=96)
    assert A.attn_fwd_workspace_size(bad) == 0


def test_resolve_3hd_gqa_offsets(lib):
    """3HD with Hq=32, Hkv=8, D=128: K at Hq*D elements, V at (Hq+Hkv)*D, token
    stride (Hq+2*Hkv)*D; the gradient buffer is resolved the same way."""
    p = params(layout="3HD", Hq=32, Hkv=8)
    r = A.attn_resolve_layout(p, FAKE * 2, None, None)
    assert r.k - r.q == 32 * 128 * 2
    assert r.v - r.q == (32 + 8) * 128 * 2
    assert r.q_token_stride == r.k_token_stride == r.v_token_stride == 48 * 128
    assert r.dk - r.dq == 32 * 128 * 2 and r.dv - r.dq == 40 * 128 * 2


def test_resolve_kv_packed_uses_v_head_dim(lib):
    """HD_2HD: V starts Hkv * v_head_dim elements after K (the corrected stride)."""
    p = params(layout="HD_2HD", Hq=64, Hkv=8, d_qk=128, d_v=128)
    r = A.attn_resolve_layout(p, FAKE * 2, FAKE * 3, None)
    assert r.v - r.k == 8 * 128 * 2
    assert r.k_token_stride == r.v_token_stride == 2 * 8 * 128
    assert r.q_token_stride == 64 * 128
    assert r.dv - r.dk == 8 * 128 * 2


@pytest.mark.parametrize("kw,code", [
    (dict(layout="3HD", Sq=256, Skv=384), 3),          # 3HD needs Sq == Skv
    (dict(layout="HD_2HD", d_qk=192, d_v=128), 3),     # KV-packed needs equal head dims
    (dict(d_qk=96), 2),                                 # unsupported head dim
    (dict(Hq=6, Hkv=4), 1),                             # Hq not a multiple of Hkv
    (dict(Hq=512, Hkv=8), 2),                           # more query heads than supported
    (dict(B=0), 1),
    (dict(scale=0.0), 1),
])
def test_validation_codes(lib, kw, code):
    p = params(**kw)
    r = A.attn_resolved_t()
    assert lib.attn_resolve_layout(ctypes.byref(p), None, None, None, ctypes.byref(r)) == code


def test_segment_shape_agreement(lib):
    """ids and pos must carry the same shape (the batcher bug of the pages:
    ids with an extra leading dim, pos without)."""
    p = params(fmt="THD_SEGMENTS")
    p.q_seg_ids = p.kv_seg_ids = FAKE
    p.q_seg_pos = p.kv_seg_pos = FAKE
    for arr in (p.q_ids_dims, p.kv_ids_dims, p.q_pos_dims, p.kv_pos_dims):
        arr[0], arr[1] = 2, 256
    r = A.attn_resolved_t()
    assert lib.attn_resolve_layout(ctypes.byref(p), None, None, None, ctypes.byref(r)) == 0
    p.q_pos_dims[0] = 1  # pos [1,256] against ids [2,256]
    assert lib.attn_resolve_layout(ctypes.byref(p), None, None, None, ctypes.byref(r)) == 3
    p.q_pos_dims[0] = 2
    p.kv_ids_dims[1] = 255
    assert lib.attn_resolve_layout(ctypes.byref(p), None, None, None, ctypes.byref(r)) == 3


def test_fwd_rejects_before_launch(lib):
    """Invalid calls return a status without touching the device."""
    p = params()
    ws_need = A.attn_fwd_workspace_size(p)
    s = lib.attn_fwd(ctypes.byref(p), ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE),
                     ctypes.c_void_p(FAKE * 4), ctypes.c_size_t(ws_need - 256), None)
    assert s == 4
    s = lib.attn_fwd(ctypes.byref(p), ctypes.c_void_p(FAKE + 8), ctypes.c_void_p(FAKE),
                     ctypes.c_void_p(FAKE * 4), ctypes.c_size_t(ws_need), None)
    assert s == 1  # misaligned output
    s = lib.attn_bwd(ctypes.byref(p), ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE),
                     ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE),
                     ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE * 4),
                     ctypes.c_size_t(A.attn_bwd_workspace_size(p)), None)
    assert s == 1  # dbias without a bias
    assert lib.attn_status_string(6) == b"device-side wait timed out"


def _bwd(lib, p, dbias=None):
    return lib.attn_bwd(ctypes.byref(p), ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE),
                        ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE),
                        ctypes.c_void_p(FAKE), dbias, ctypes.c_void_p(FAKE * 4),
                        ctypes.c_size_t(A.attn_bwd_workspace_size(p)), None)


def test_params_version_checked(lib):
    p = params()
    p.struct_version = A.ATTN_PARAMS_VERSION - 1
    r = A.attn_resolved_t()
    assert lib.attn_resolve_layout(ctypes.byref(p), None, None, None, ctypes.byref(r)) == 1
    assert lib.attn_abi_version() == A.ATTN_PARAMS_VERSION


def test_max_logit_and_sink_arguments_checked(lib):
    """Optional max-logit / sink / dsink pointers: misaligned ones and a sink
    gradient without sink logits are rejected before any launch."""
    p = params()
    ws_need = A.attn_fwd_workspace_size(p)

    def fwd():
        return lib.attn_fwd(ctypes.byref(p), ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE),
                            ctypes.c_void_p(FAKE * 4), ctypes.c_size_t(ws_need), None)

    p.max_logit = FAKE + 2
    assert fwd() == 1
    p.max_logit = None
    p.sink = FAKE + 1
    assert fwd() == 1
    p.sink = None
    p.dsink = FAKE
    assert _bwd(lib, p) == 1  # a sink gradient needs sink logits
    p.sink = FAKE + 2
    assert _bwd(lib, p) == 1  # misaligned sink
    p.sink = FAKE
    p.dsink = FAKE + 6
    assert _bwd(lib, p) == 1  # misaligned dsink


def test_sink_gradient_workspace(lib):
    """The sink gradient needs one partial per preprocess block (8 tokens) and
    query head in the backward workspace."""
    p = params()
    base = A.attn_bwd_workspace_size(p)
    p.sink, p.dsink = FAKE, FAKE
    need = (2 * 256 + 7) // 8 * 8 * 4
    assert A.attn_bwd_workspace_size(p) - base == (need + 255) // 256 * 256
    assert A.attn_fwd_workspace_size(p) == A.attn_fwd_workspace_size(params())


def test_band_validation(lib):
    """A causal mask keeps at most the diagonal on the right: a band that
    reaches past it is rejected; an open or zero right side is accepted, as
    is any band without a causal mask."""
    p = params(mask="CAUSAL")
    p.band, p.window_left, p.window_right = 1, 100, 5
    assert A.attn_fwd_workspace_size(p) == 0
    for right in (0, -1):
        p.window_right = right
        assert A.attn_fwd_workspace_size(p) > 0
    q = params(mask="NONE")
    q.band, q.window_left, q.window_right, q.bottom_right = 1, -1, 7, 1
    assert A.attn_fwd_workspace_size(q) > 0
    m = A.make_params(layout="HD_HD_HD", fmt="BSHD", mask="CAUSAL", B=1, Sq=8, Skv=8, Hq=1,
                      Hkv=1, d_qk=64, d_v=64, scale=0.1, q=None, window=(None, 0),
                      bottom_right=True)
    assert (m.band, m.window_left, m.window_right, m.bottom_right) == (1, -1, 0, 1)


def test_dtype_validation(lib):
    p = params()
    p.descale_q = p.descale_k = p.descale_v = 1.0
    for dt, ok in ((0, True), (1, True), (2, True), (3, False), (-1, False)):
        p.dtype = dt
        assert (A.attn_fwd_workspace_size(p) > 0) == ok


def test_fp8_forward_validation(lib):
    """E4M3 forward: descale factors positive and finite (INVALID_ARG),
    head dims 128 and no bias or sink (UNSUPPORTED), forward only (the
    backward and the no-allocation entry point return UNSUPPORTED), and a
    workspace that holds the transposed V planes."""
    def fp8(**kw):
        p = params(**kw)
        p.dtype = 2
        p.descale_q, p.descale_k, p.descale_v = 0.5, 2.0, 1.0
        return p

    p = fp8()
    assert lib.attn_fwd_workspace_size(ctypes.byref(p)) > 0
    pb = params()
    # one byte per element of V^T: B * Hkv * d_v * (Skv rounded to 128, plus 128)
    assert (A.attn_fwd_workspace_size(p) - A.attn_fwd_workspace_size(pb)
            >= 2 * 2 * 128 * (256 + 128))
    for field, val in (("descale_q", 0.0), ("descale_k", -1.0), ("descale_v", float("inf")),
                       ("descale_v", float("nan"))):
        q = fp8()
        setattr(q, field, val)
        assert A.attn_fwd_workspace_size(q) == 0, field
        assert lib.attn_resolve_layout(ctypes.byref(q), None, None, None,
                                       ctypes.byref(A.attn_resolved_t())) == 1
    r = A.attn_resolved_t()
    assert lib.attn_resolve_layout(ctypes.byref(fp8(d_qk=64, d_v=64)), None, None, None,
                                   ctypes.byref(r)) == 2
    q = fp8()
    q.bias = FAKE
    q.bias_b, q.bias_h = 1, 8
    assert lib.attn_resolve_layout(ctypes.byref(q), None, None, None, ctypes.byref(r)) == 2
    assert _bwd(lib, fp8()) == 2
    assert lib.attn_fwd_noalloc(ctypes.byref(fp8()), ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE),
                                None) == 2
    # packed layouts resolve with one-byte elements
    q = fp8(layout="3HD")
    assert lib.attn_resolve_layout(ctypes.byref(q), None, None, None, ctypes.byref(r)) == 0
    assert r.k - r.q == 8 * 128 and r.v - r.q == (8 + 2) * 128
    assert r.q_token_stride == (8 + 2 + 2) * 128
    m = A.make_params(layout="HD_HD_HD", fmt="BSHD", mask="NONE", B=1, Sq=8, Skv=8, Hq=1, Hkv=1,
                      d_qk=64, d_v=64, scale=0.1, q=None, dtype="fp16")
    assert m.dtype == 1
