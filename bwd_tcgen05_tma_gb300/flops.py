"""Exact algorithmic FLOP counts of fused attention from the segment metadata.

The count of unmasked (query, key) pairs P is exact for the given metadata;
forward = 2 P (d_qk + d_v), backward = 2 P (3 d_qk + 2 d_v) (the five GEMMs
S = QK^T recomputed, dP = dO V^T, dV, dK, dQ).  Tile waste and the two extra
GEMMs of the deterministic dQ pass are not credited.
"""
from __future__ import annotations

import numpy as np


def _row_pairs(id_q, pos_q, id_kv, pos_kv, causal):
    total = 0
    for u in np.unique(id_q):
        if u == 0:
            continue
        kv_sel = id_kv == u
        if not kv_sel.any():
            continue
        q_sel = id_q == u
        if not causal:
            total += int(q_sel.sum()) * int(kv_sel.sum())
        else:
            pk = np.sort(pos_kv[kv_sel])
            total += int(np.searchsorted(pk, pos_q[q_sel], side="right").sum())
    return total


def _derive_pos(ids):
    pos = np.zeros_like(ids)
    for b in range(ids.shape[0]):
        starts = np.r_[True, ids[b, 1:] != ids[b, :-1]]
        idx = np.arange(ids.shape[1])
        run_start = np.maximum.accumulate(np.where(starts, idx, 0))
        pos[b] = idx - run_start
    return pos


def valid_pairs_per_head(case):
    """Exact number of unmasked pairs summed over batch rows, for one head."""
    if case.fmt == "BSHD" and case.q_ids is None:
        if not case.causal:
            return case.B * case.Sq * case.Skv
        n = min(case.Sq, case.Skv)
        # top-left causal: row i sees keys 0..i
        rows = np.arange(case.Sq)
        return case.B * int(np.minimum(rows + 1, case.Skv).sum()) if n else 0
    if case.fmt == "THD_CU_SEQLENS":
        cq, ck = np.asarray(case.cu_seqlens_q), np.asarray(case.cu_seqlens_kv)
        total = 0
        for k in range(len(cq) - 1):
            lq, lk = int(cq[k + 1] - cq[k]), int(ck[k + 1] - ck[k])
            if case.causal:
                total += int(np.minimum(np.arange(lq) + 1, lk).sum())
            else:
                total += lq * lk
        return total
    qp = case.q_pos if case.q_pos is not None else _derive_pos(case.q_ids)
    kp = case.kv_pos if case.kv_pos is not None else _derive_pos(case.kv_ids)
    return sum(_row_pairs(case.q_ids[b], qp[b], case.kv_ids[b], kp[b], case.causal)
               for b in range(case.B))


def attention_flops(case):
    """(forward FLOPs, backward FLOPs, unmasked pairs over all heads)."""
    P = valid_pairs_per_head(case) * case.Hq
    return 2.0 * P * (case.d_qk + case.d_v), 2.0 * P * (3 * case.d_qk + 2 * case.d_v), P
