import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workload")


def oracle_metadata(case):
    """Per-token (ids, pos) for Q and KV in the oracle's terms."""
    from oracle import attn_ref as R

    if case.fmt == "BSHD" and case.q_ids is None:
        qi, qp = R.dense_metadata(case.B, case.Sq)
        ki, kp = R.dense_metadata(case.B, case.Skv)
        return qi, qp, ki, kp
    if case.fmt == "THD_CU_SEQLENS":
        qi, qp = R.metadata_from_cu_seqlens(case.cu_seqlens_q, case.Sq)
        ki, kp = R.metadata_from_cu_seqlens(case.cu_seqlens_kv, case.Skv)
        return qi, qp, ki, kp
    qp = case.q_pos if case.q_pos is not None else R.derive_segment_pos(case.q_ids)
    kp = case.kv_pos if case.kv_pos is not None else R.derive_segment_pos(case.kv_ids)
    return case.q_ids, qp, case.kv_ids, kp


def oracle_mask(case):
    """The oracle's mask argument for a case: the causal flag, or a Window
    when the case has a band or bottom-right alignment (a causal mask keeps
    the band's right side at 0)."""
    from oracle import attn_ref as R

    if case.window is None and not case.bottom_right:
        return case.causal
    left, right = case.window if case.window is not None else (None, None)
    if case.causal:
        right = 0
    shift = case.Skv - case.Sq if case.bottom_right else 0
    return R.Window(left, right, shift)


def oracle_qkv(case):
    from oracle import attn_ref as R

    return R.unpack_layout(case.layout, case.buffers, case.B, case.Sq, case.Skv, case.Hq,
                           case.Hkv, case.d_qk, case.d_v)


def oracle_full(case):
    """Full oracle forward + backward of a case: dict of float64 arrays."""
    from oracle import attn_ref as R

    q, k, v = oracle_qkv(case)
    qi, qp, ki, kp = oracle_metadata(case)
    bias = None if case.bias is None else case.bias.astype(np.float64)
    mask = oracle_mask(case)
    o, lse = R.attention_forward(q, k, v, qi, qp, ki, kp, mask, case.scale, bias)
    dq, dk, dv, dbias = R.attention_backward(q, k, v, case.do.astype(np.float64), qi, qp, ki,
                                             kp, mask, case.scale, bias)
    return {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv, "dbias": dbias}


@pytest.fixture
def rng():
    return np.random.default_rng(1234)
