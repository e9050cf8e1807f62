"""Helpers for GPU parity tests: move a seeded case to the device, call the
library through the C ABI, and compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

from bwd_tcgen05_tma_gb300 import attn as A
from bwd_tcgen05_tma_gb300 import inputs as I

# tolerances (relative Frobenius error)
TOL_O = 5e-3
TOL_LSE = 5e-3
TOL_GRAD = 1.5e-2
TOL_DBIAS = 3e-2


def bf16_dev(x, dtype="bf16"):
    """A float32 array holding values of the element type -> device tensor of
    that type (exact: the values are representable)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "fp16":
        return torch.from_numpy(x.astype(np.float16)).cuda()
    bits = I.bf16_bits(x)
    return torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)


def torch_dtype(case):
    return torch.float16 if case.dtype == "fp16" else torch.bfloat16


def int_dev(x):
    return None if x is None else torch.from_numpy(np.ascontiguousarray(x, dtype=np.int32)).cuda()


class DevCase:
    """Device copies of one case plus its parameter block."""

    def __init__(self, case, dq_mode="deterministic", force_general=False, with_pos=True):
        self.case = c = case
        self.t = {k: bf16_dev(v, c.dtype) for k, v in c.buffers.items()}
        self.do = bf16_dev(c.do.reshape(c.B * c.Sq, c.Hq, c.d_v), c.dtype)
        self.bias = bf16_dev(c.bias, c.dtype) if c.bias is not None else None
        self.q_ids = int_dev(c.q_ids)
        self.kv_ids = int_dev(c.kv_ids)
        self.q_pos = int_dev(c.q_pos) if with_pos else None
        self.kv_pos = int_dev(c.kv_pos) if with_pos else None
        self.cu_q = int_dev(c.cu_seqlens_q)
        self.cu_kv = int_dev(c.cu_seqlens_kv)
        if c.layout == "3HD":
            q, k, v = self.t["qkv"], None, None
        elif c.layout == "HD_2HD":
            q, k, v = self.t["q"], self.t["kv"], None
        else:
            q, k, v = self.t["q"], self.t["k"], self.t["v"]
        self.params = A.make_params(
            layout=c.layout, fmt=c.fmt, mask=c.mask, B=c.B, Sq=c.Sq, Skv=c.Skv, Hq=c.Hq,
            Hkv=c.Hkv, d_qk=c.d_qk, d_v=c.d_v, scale=c.scale, q=q, k=k, v=v,
            q_seg_ids=self.q_ids, q_seg_pos=self.q_pos, kv_seg_ids=self.kv_ids,
            kv_seg_pos=self.kv_pos, cu_seqlens_q=self.cu_q, cu_seqlens_kv=self.cu_kv,
            bias=self.bias, dq_mode=dq_mode, force_general_path=force_general,
            window=c.window, bottom_right=c.bottom_right, dtype=c.dtype)
        self.ws_fwd = torch.zeros(max(A.attn_fwd_workspace_size(self.params), 256),
                                  dtype=torch.uint8, device="cuda")
        self.ws_bwd = torch.zeros(max(A.attn_bwd_workspace_size(self.params), 256),
                                  dtype=torch.uint8, device="cuda")

    def forward(self, canary=True):
        c = self.case
        fill = float("nan") if canary else 0.0
        self.o = torch.full((c.B * c.Sq, c.Hq, c.d_v), fill, dtype=torch_dtype(c), device="cuda")
        self.lse = torch.full((c.B, c.Hq, c.Sq), fill, dtype=torch.float32, device="cuda")
        A.attn_fwd(self.params, self.o, self.lse, self.ws_fwd)
        st, stats = A.attn_read_status(self.ws_fwd)
        assert st == 0, f"device status {st}"
        self.fwd_stats = stats
        return self.o, self.lse

    def grad_buffers(self, canary=True):
        c = self.case
        fill = float("nan") if canary else 0.0

        def z(*shape):
            return torch.full(shape, fill, dtype=torch_dtype(c), device="cuda")

        if c.layout == "3HD":
            W = c.Hq * c.d_qk + c.Hkv * c.d_qk + c.Hkv * c.d_v
            g = {"dqkv": z(c.B * c.Sq, W)}
            return g, (g["dqkv"], None, None)
        if c.layout == "HD_2HD":
            g = {"dq": z(c.B * c.Sq, c.Hq * c.d_qk), "dkv": z(c.B * c.Skv, 2, c.Hkv, c.d_v)}
            return g, (g["dq"], g["dkv"], None)
        g = {"dq": z(c.B, c.Sq, c.Hq, c.d_qk), "dk": z(c.B, c.Skv, c.Hkv, c.d_qk),
             "dv": z(c.B, c.Skv, c.Hkv, c.d_v)}
        return g, (g["dq"], g["dk"], g["dv"])

    def backward(self, canary=True, want_dbias=True):
        c = self.case
        g, (dq, dk, dv) = self.grad_buffers(canary)
        dbias = None
        if c.bias is not None and want_dbias:
            dbias = torch.full(c.bias.shape, float("nan") if canary else 0.0,
                               dtype=torch_dtype(c), device="cuda")
        A.attn_bwd(self.params, self.o, self.do, self.lse, dq, dk, dv, dbias, self.ws_bwd)
        st, stats = A.attn_read_status(self.ws_bwd)
        assert st == 0, f"device status {st}"
        self.bwd_stats = stats
        self.grads = g
        self.dbias = dbias
        return g, dbias


def unpack_grads(case, g):
    """Device gradient buffers -> float64 dQ [B,Sq,Hq,dqk], dK, dV."""
    from oracle import attn_ref as R

    host = {k: v.float().cpu().numpy() for k, v in g.items()}
    B, Sq, Skv, Hq, Hkv, dqk, dv = (case.B, case.Sq, case.Skv, case.Hq, case.Hkv, case.d_qk,
                                    case.d_v)
    if case.layout == "3HD":
        return R.unpack_layout("3HD", {"qkv": host["dqkv"]}, B, Sq, Skv, Hq, Hkv, dqk, dv)
    if case.layout == "HD_2HD":
        return R.unpack_layout("HD_2HD", {"q": host["dq"], "kv": host["dkv"]}, B, Sq, Skv, Hq,
                               Hkv, dqk, dv)
    return (host["dq"].astype(np.float64), host["dk"].astype(np.float64),
            host["dv"].astype(np.float64))


def rel(x, ref):
    from oracle import attn_ref as R

    return R.rel_frobenius(x, ref)


def check_forward(case, ref, o_dev, lse_dev):
    """O and LSE against the oracle; rows without keys must be exactly 0 / -inf."""
    o = o_dev.float().cpu().numpy().reshape(case.B, case.Sq, case.Hq, case.d_v)
    lse = lse_dev.cpu().numpy()
    has = np.isfinite(ref["lse"])  # [B,Hq,Sq]
    assert np.array_equal(np.isfinite(lse), has), "LSE finiteness pattern differs"
    assert np.all(np.isneginf(lse[~has]))
    has_o = has.transpose(0, 2, 1)  # [B,Sq,Hq]
    assert np.all(o[~has_o] == 0.0), "rows without keys must give O = 0"
    eo = rel(o[has_o], ref["o"][has_o])
    el = rel(lse[has], ref["lse"][has])
    assert eo <= TOL_O, f"O rel err {eo}"
    assert el <= TOL_LSE, f"LSE rel err {el}"
    return eo, el


def structural_masks(case):
    """Per batch row: valid-pair matrix, queries without keys, keys without queries."""
    from conftest import oracle_mask, oracle_metadata
    from oracle import attn_ref as R

    qi, qp, ki, kp = oracle_metadata(case)
    mask = oracle_mask(case)
    valid = np.stack([R.valid_pairs(qi[b], qp[b], ki[b], kp[b], mask)
                      for b in range(case.B)])
    return valid, ~valid.any(axis=2), ~valid.any(axis=1)


def check_backward(case, ref, grads, dbias_dev):
    dq, dk, dv = unpack_grads(case, grads)
    valid, q_dead, k_dead = structural_masks(case)
    out = {}
    for name, x, r, dead in (("dq", dq, ref["dq"], q_dead), ("dk", dk, ref["dk"], k_dead),
                             ("dv", dv, ref["dv"], k_dead)):
        assert np.all(np.isfinite(x)), f"{name} has non-finite values (unwritten elements?)"
        e = rel(x, r)
        out[name] = e
        assert e <= TOL_GRAD, f"{name} rel err {e}"
        assert np.all(x[dead] == 0.0), f"{name}: tokens without a valid pair must get exactly 0"
    if dbias_dev is not None:
        db = dbias_dev.float().cpu().numpy()
        assert np.all(np.isfinite(db))
        e = rel(db, ref["dbias"])
        out["dbias"] = e
        assert e <= TOL_DBIAS, f"dbias rel err {e}"
        # pairs that are invalid in every (batch row, head) summed into an element
        inval_all = ~valid.any(axis=0) if db.shape[0] == 1 else ~valid
        inval = np.broadcast_to(inval_all[:, None] if inval_all.ndim == 3 else inval_all[None, None],
                                db.shape)
        assert np.all(db[inval] == 0.0), "dBias must be exactly 0 at masked pairs"
    return out
