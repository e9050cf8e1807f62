"""Pins for the two oracle functions every measurement rests on (CPU only):

* ``rel_frobenius``, the parity metric of every GPU test, against values
  worked out by hand;
* ``attention_flops``, the numerator of the CPU baseline and of the reference
  arm, against an attention computed with scalar loops that counts every
  multiply and add it performs, and against the FLOP figures of the dense
  causal workload (B=4, S=2048, 16 heads, D=128: 2,098,176 pairs per row and
  head, 68.8 GFLOP forward, 171.9 GFLOP backward).

Each function also gets planted mistakes (in a copy of the oracle) that these
pins must catch.
"""
import inspect
import math
import types

import numpy as np
import pytest

from oracle import attn_ref as R


def _mutant(old, new):
    src = inspect.getsource(R)
    assert src.count(old) == 1, old
    mod = types.ModuleType("oracle_mutant")
    exec(compile(src.replace(old, new, 1), "oracle_mutant", "exec"), mod.__dict__)
    return mod


# ----------------------------------------------------------------- rel_frobenius


def _frobenius_pins(f):
    """Hand-computed cases; returns the list of those that fail."""
    bad = []
    ref = np.array([[1.0, -2.0], [3.0, 0.5]])
    if f(ref, ref) != 0.0:
        bad.append("x == ref gives 0")
    if not math.isclose(f(2.0 * ref, ref), 1.0, rel_tol=1e-15):
        bad.append("x = 2 ref gives 1")
    if not math.isclose(f(np.zeros(2), np.array([3.0, 4.0])), 1.0, rel_tol=1e-15):
        bad.append("x = 0 gives 1")
    # ||(0, 2, 2)|| / ||(1, 0, 0)|| = sqrt(8)
    if not math.isclose(f(np.array([1.0, 2.0, 2.0]), np.array([1.0, 0.0, 0.0])), 2.0 * math.sqrt(2.0),
                        rel_tol=1e-15):
        bad.append("2 sqrt 2 case")
    # ||(3, 4) - (0, 4)|| / ||(0, 4)|| = 3 / 4, while ||x|| = 5
    if not math.isclose(f(np.array([3.0, 4.0]), np.array([0.0, 4.0])), 0.75, rel_tol=1e-15):
        bad.append("divides by ||ref||")
    if f(np.array([3.0, 4.0]), np.zeros(2)) != math.inf:
        bad.append("nonzero x against zero ref gives inf")
    if f(np.zeros(3), np.zeros(3)) != 0.0:
        bad.append("both zero gives 0")
    return bad


def test_rel_frobenius_hand_values():
    assert _frobenius_pins(R.rel_frobenius) == []


@pytest.mark.parametrize("old,new", [
    # no square roots: ratio of squared norms
    ("den = np.linalg.norm(ref.ravel())", "den = float((ref.ravel() ** 2).sum())"),
    # divides by ||x|| instead of ||ref||
    ("den = np.linalg.norm(ref.ravel())", "den = np.linalg.norm(x.ravel())"),
    # a zero reference always passes
    ("return 0.0 if num == 0.0 else np.inf", "return 0.0"),
    # absolute instead of relative error
    ("return float(num / den)", "return float(num)"),
])
def test_rel_frobenius_planted_mistakes_caught(old, new):
    with np.errstate(all="ignore"):
        assert _frobenius_pins(_mutant(old, new).rel_frobenius) != []


# ----------------------------------------------------------------- attention_flops


def counted_attention(q, k, v, do, valid, scale):
    """Forward and backward of one head with scalar loops over the valid pairs,
    counting one FLOP per scalar multiply and one per scalar add of the five
    backward products (S recomputed, dP, dV, dK, dQ) and the two forward ones
    (S, P V).  The softmax itself (exp, max, sums) is not a matrix product and
    is not counted.  Returns (O, dQ, dK, dV, forward FLOPs, backward FLOPs)."""
    Sq, dk = q.shape
    Skv, dv = v.shape
    fl_f = fl_b = 0

    def dot(a, b):
        acc = 0.0
        for c in range(len(a)):
            acc += a[c] * b[c]
        return acc, 2 * len(a)  # one multiply and one add per element

    s = np.full((Sq, Skv), -np.inf)
    for i in range(Sq):
        for j in range(Skv):
            if valid[i, j]:
                s[i, j], n = dot(q[i], k[j])
                s[i, j] *= scale
                fl_f += n
    p = np.zeros((Sq, Skv))
    o = np.zeros((Sq, dv))
    for i in range(Sq):
        if valid[i].any():
            m = s[i][valid[i]].max()
            e = np.where(valid[i], np.exp(s[i] - m), 0.0)
            p[i] = e / e.sum()
        for j in range(Skv):
            if valid[i, j]:
                for c in range(dv):
                    o[i, c] += p[i, j] * v[j, c]
                fl_f += 2 * dv
    dq = np.zeros_like(q)
    dkk = np.zeros_like(k)
    dvv = np.zeros_like(v)
    for i in range(Sq):
        D, _ = dot(do[i], o[i])
        for j in range(Skv):
            if not valid[i, j]:
                continue
            _, n = dot(q[i], k[j])  # S recomputed
            fl_b += n
            dp, n = dot(do[i], v[j])
            fl_b += n
            for c in range(dv):
                dvv[j, c] += p[i, j] * do[i, c]
            fl_b += 2 * dv
            ds = p[i, j] * (dp - D)
            for c in range(dk):
                dq[i, c] += scale * ds * k[j, c]
                dkk[j, c] += scale * ds * q[i, c]
            fl_b += 2 * dk + 2 * dk
    return o, dq, dkk, dvv, fl_f, fl_b


@pytest.mark.parametrize("dk,dv,causal", [(5, 3, True), (3, 7, False), (4, 4, True)])
def test_attention_flops_matches_counted_loops(dk, dv, causal):
    """The counted scalar-loop attention computes what the oracle computes (so
    the loops are a real attention), and attention_flops on its pair count
    equals the FLOPs those loops performed."""
    rng = np.random.default_rng(3 + dk)
    Sq = Skv = 9
    ids = np.array([[1, 1, 1, 1, 2, 2, 2, 2, 0]])
    pos = np.array([[0, 1, 2, 3, 0, 1, 2, 3, 0]])
    q = rng.standard_normal((1, Sq, 1, dk))
    k = rng.standard_normal((1, Skv, 1, dk))
    v = rng.standard_normal((1, Skv, 1, dv))
    do = rng.standard_normal((1, Sq, 1, dv))
    scale = 0.37
    valid = R.valid_pairs(ids[0], pos[0], ids[0], pos[0], causal)
    o, dq, dkk, dvv, fl_f, fl_b = counted_attention(q[0, :, 0], k[0, :, 0], v[0, :, 0],
                                                     do[0, :, 0], valid, scale)
    ro, _ = R.attention_forward(q, k, v, ids, pos, ids, pos, causal, scale)
    rdq, rdk, rdv, _ = R.attention_backward(q, k, v, do, ids, pos, ids, pos, causal, scale)
    np.testing.assert_allclose(o, ro[0, :, 0], atol=1e-12)
    np.testing.assert_allclose(dq, rdq[0, :, 0], atol=1e-12)
    np.testing.assert_allclose(dkk, rdk[0, :, 0], atol=1e-12)
    np.testing.assert_allclose(dvv, rdv[0, :, 0], atol=1e-12)
    pairs = R.count_valid_pairs(ids, pos, ids, pos, causal)
    assert pairs == int(valid.sum())
    assert R.attention_flops(pairs, dk, dv) == (fl_f, fl_b)


def test_attention_flops_dense_causal_workload():
    """Dense causal B=4, S=2048, 16 heads, D=128: each row and head has
    2048 * 2049 / 2 = 2,098,176 pairs, P = 134,283,264 in all; forward
    68,753,031,168 FLOPs, backward 171,882,577,920."""
    P = 2048 * 2049 // 2 * 4 * 16
    assert P == 134_283_264
    ids, pos = R.dense_metadata(1, 2048)
    assert R.count_valid_pairs(ids, pos, ids, pos, True) == 2_098_176
    assert R.attention_flops(P, 128, 128) == (68_753_031_168, 171_882_577_920)


@pytest.mark.parametrize("old,new", [
    ("2.0 * P * (3 * d_qk + 2 * d_v)", "2.0 * P * (2 * d_qk + 3 * d_v)"),  # dims swapped
    ("2.0 * P * (3 * d_qk + 2 * d_v)", "2.0 * P * (2 * d_qk + 2 * d_v)"),  # S recompute dropped
    ("return 2.0 * P * (d_qk + d_v)", "return P * (d_qk + d_v)"),  # multiply-adds as one FLOP
])
def test_attention_flops_planted_mistakes_caught(old, new):
    bad = _mutant(old, new).attention_flops
    caught = bad(134_283_264, 128, 128) != (68_753_031_168, 171_882_577_920)
    ids = np.array([[1, 1, 1, 1, 2, 2, 2, 2, 0]])
    pos = np.array([[0, 1, 2, 3, 0, 1, 2, 3, 0]])
    valid = R.valid_pairs(ids[0], pos[0], ids[0], pos[0], True)
    rng = np.random.default_rng(0)
    *_, fl_f, fl_b = counted_attention(rng.standard_normal((9, 5)), rng.standard_normal((9, 5)),
                                       rng.standard_normal((9, 3)), rng.standard_normal((9, 3)),
                                       valid, 0.5)
    caught = caught or bad(int(valid.sum()), 5, 3) != (fl_f, fl_b)
    assert caught
