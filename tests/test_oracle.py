"""Pins for the float64 oracle (CPU only).

Each test checks the oracle against something other than itself: a library
routine (torch SDPA / autograd in float64), central finite differences, closed
forms, invariants, or brute-force scalar loops.  The mutation tests at the end
plant plausible mistakes in a copy of the oracle and check that the pins catch
every one of them.
"""
import math
import types

import numpy as np
import pytest
import torch

from oracle import attn_ref as R


# ----------------------------------------------------------------- helpers


def rand(rng, *shape):
    return rng.standard_normal(shape)


def seg_meta(lens_per_row, S):
    """ids/pos [B,S] from per-row segment length lists (tail is padding)."""
    B = len(lens_per_row)
    ids = np.zeros((B, S), np.int64)
    pos = np.zeros((B, S), np.int64)
    for b, lens in enumerate(lens_per_row):
        t = 0
        for k, L in enumerate(lens):
            ids[b, t:t + L] = k + 1
            pos[b, t:t + L] = np.arange(L)
            t += L
    return ids, pos


def brute_force(q, k, v, do, idq, posq, idk, posk, causal, scale, bias=None, sink=None):
    """Pure-Python scalar loops (no BLAS).  D is taken as the row sum of
    dO * O, the other form of the identity the oracle's D uses.  With sink
    logits each row's normaliser also holds exp(sink_h - m)."""
    B, Sq, Hq, Dk = q.shape
    _, Skv, Hkv, Dv = v.shape
    grp = Hq // Hkv
    o = np.zeros((B, Sq, Hq, Dv))
    lse = np.full((B, Hq, Sq), -np.inf)
    dq = np.zeros(q.shape)
    dk = np.zeros(k.shape)
    dv = np.zeros(v.shape)
    dbias = None if bias is None else np.zeros(bias.shape)
    for b in range(B):
        for h in range(Hq):
            g = h // grp
            bb = b if (bias is not None and bias.shape[0] > 1) else 0
            bh = h if (bias is not None and bias.shape[1] > 1) else 0
            for i in range(Sq):
                valid = []
                s = []
                for j in range(Skv):
                    ok = idq[b, i] == idk[b, j] and idq[b, i] != 0
                    if isinstance(causal, tuple):  # (left, right, shift) band
                        left, right, shift = causal
                        rel = posk[b, j] - (posq[b, i] + shift)
                        ok = ok and (left is None or rel >= -left) and (right is None or rel <= right)
                    elif causal:
                        ok = ok and posk[b, j] <= posq[b, i]
                    if ok:
                        acc = 0.0
                        for c in range(Dk):
                            acc += q[b, i, h, c] * k[b, j, g, c]
                        acc *= scale
                        if bias is not None:
                            acc += bias[bb, bh, i, j]
                        valid.append(j)
                        s.append(acc)
                if not valid:
                    if sink is not None:
                        lse[b, h, i] = sink[h]
                    continue
                m = max(s) if sink is None else max(max(s), sink[h])
                e = [math.exp(x - m) for x in s]
                l = sum(e) + (0.0 if sink is None else math.exp(sink[h] - m))
                p = [x / l for x in e]
                lse[b, h, i] = m + math.log(l)
                for c in range(Dv):
                    o[b, i, h, c] = sum(p[t] * v[b, j, g, c] for t, j in enumerate(valid))
                Di = sum(do[b, i, h, c] * o[b, i, h, c] for c in range(Dv))
                for t, j in enumerate(valid):
                    dp = sum(do[b, i, h, c] * v[b, j, g, c] for c in range(Dv))
                    ds = p[t] * (dp - Di)
                    for c in range(Dk):
                        dq[b, i, h, c] += scale * ds * k[b, j, g, c]
                        dk[b, j, g, c] += scale * ds * q[b, i, h, c]
                    for c in range(Dv):
                        dv[b, j, g, c] += p[t] * do[b, i, h, c]
                    if dbias is not None:
                        dbias[bb, bh, i, j] += ds
    return o, lse, dq, dk, dv, dbias


def small_problem(rng, *, B=2, S=11, Skv=None, Hq=4, Hkv=2, Dk=5, Dv=3, causal=True,
                  with_bias=True, bias_shape=None, cross=False):
    Skv = S if Skv is None else Skv
    q = rand(rng, B, S, Hq, Dk)
    k = rand(rng, B, Skv, Hkv, Dk)
    v = rand(rng, B, Skv, Hkv, Dv)
    do = rand(rng, B, S, Hq, Dv)
    idq, posq = seg_meta([[4, 5], [7, 2]], S)  # rows end with padding tails
    if cross:
        idk, posk = seg_meta([[3, 6, 2], [5, 4]], Skv)
    else:
        idk, posk = idq.copy(), posq.copy()
    bias = None
    if with_bias:
        shp = bias_shape or (1, Hq, S, Skv)
        bias = 0.5 * rand(rng, *shp)
    return q, k, v, do, idq, posq, idk, posk, causal, 0.7, bias


def run_oracle(mod, prob):
    q, k, v, do, idq, posq, idk, posk, causal, scale, bias = prob
    o, lse = mod.attention_forward(q, k, v, idq, posq, idk, posk, causal, scale, bias,
                                   row_block=4)
    dq, dk, dv, db = mod.attention_backward(q, k, v, do, idq, posq, idk, posk, causal, scale,
                                            bias, row_block=4)
    return o, lse, dq, dk, dv, db


def assert_same(a, b, tol=1e-10):
    if a is None or b is None:
        assert a is None and b is None
        return
    fin = np.isfinite(b)
    assert np.array_equal(np.isfinite(a), fin)
    assert np.allclose(a[fin], b[fin], rtol=tol, atol=tol)


# ----------------------------------------------------------------- pins


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("cross", [False, True])
def test_brute_force_scalar_loops(rng, causal, cross):
    prob = small_problem(rng, causal=causal, cross=cross, S=9, Skv=12 if cross else None)
    got = run_oracle(R, prob)
    ref = brute_force(*prob)
    for a, b in zip(got, ref):
        assert_same(a, b)


@pytest.mark.parametrize("bias_shape", [(2, 4, 11, 11), (1, 4, 11, 11), (2, 1, 11, 11),
                                        (1, 1, 11, 11)])
def test_bias_broadcast_reduction_brute(rng, bias_shape):
    prob = small_problem(rng, bias_shape=bias_shape)
    got = run_oracle(R, prob)
    ref = brute_force(*prob)
    assert_same(got[5], ref[5])


@pytest.mark.parametrize("causal", [False, True])
def test_dense_matches_torch_sdpa_and_autograd(rng, causal):
    """Unmasked, unsegmented, Hq == Hkv: forward equals torch SDPA in float64,
    gradients equal torch autograd through it."""
    B, S, H, D = 2, 37, 3, 16
    q, k, v, do = rand(rng, B, S, H, D), rand(rng, B, S, H, D), rand(rng, B, S, H, D), rand(
        rng, B, S, H, D)
    ids, pos = R.dense_metadata(B, S)
    scale = 1 / math.sqrt(D)
    o, lse = R.attention_forward(q, k, v, ids, pos, ids, pos, causal, scale, row_block=16)
    dq, dk, dv, _ = R.attention_backward(q, k, v, do, ids, pos, ids, pos, causal, scale,
                                         row_block=16)
    tq, tk, tv = (torch.tensor(x.transpose(0, 2, 1, 3), requires_grad=True) for x in (q, k, v))
    to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal,
                                                          scale=scale)
    to.backward(torch.tensor(do.transpose(0, 2, 1, 3)))
    np.testing.assert_allclose(o, to.detach().numpy().transpose(0, 2, 1, 3), rtol=1e-12,
                               atol=1e-12)
    np.testing.assert_allclose(dq, tq.grad.numpy().transpose(0, 2, 1, 3), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy().transpose(0, 2, 1, 3), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy().transpose(0, 2, 1, 3), rtol=1e-10, atol=1e-12)
    scores = scale * torch.einsum("bhid,bhjd->bhij", tq.detach(), tk.detach())
    if causal:
        scores = scores.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), -torch.inf)
    np.testing.assert_allclose(lse, torch.logsumexp(scores, -1).numpy(), rtol=1e-12)


def test_segments_gqa_bias_match_torch_autograd(rng):
    """Segments (no fully masked rows), GQA and a batch-broadcast bias against
    torch autograd: K/V heads expanded with repeat_interleave, the mask and
    bias passed as a float attention mask; autograd sums the bias gradient over
    the broadcast batch axis."""
    B, S, Hq, Hkv, D = 2, 13, 4, 2, 6
    q, k, v, do = rand(rng, B, S, Hq, D), rand(rng, B, S, Hkv, D), rand(rng, B, S, Hkv, D), rand(
        rng, B, S, Hq, D)
    ids, pos = seg_meta([[5, 8], [2, 6, 5]], S)
    bias = 0.5 * rand(rng, 1, Hq, S, S)
    scale = 0.4
    o, _ = R.attention_forward(q, k, v, ids, pos, ids, pos, True, scale, bias, row_block=5)
    dq, dk, dv, db = R.attention_backward(q, k, v, do, ids, pos, ids, pos, True, scale, bias,
                                          row_block=5)
    mask = np.stack([R.valid_pairs(ids[b], pos[b], ids[b], pos[b], True) for b in range(B)])
    tq = torch.tensor(q.transpose(0, 2, 1, 3), requires_grad=True)
    tk = torch.tensor(k.transpose(0, 2, 1, 3), requires_grad=True)
    tv = torch.tensor(v.transpose(0, 2, 1, 3), requires_grad=True)
    tb = torch.tensor(bias, requires_grad=True)
    fm = torch.where(torch.tensor(mask)[:, None], tb, torch.tensor(-torch.inf, dtype=tb.dtype))
    to = torch.nn.functional.scaled_dot_product_attention(
        tq, tk.repeat_interleave(Hq // Hkv, 1), tv.repeat_interleave(Hq // Hkv, 1),
        attn_mask=fm, scale=scale)
    to.backward(torch.tensor(do.transpose(0, 2, 1, 3)))
    np.testing.assert_allclose(o, to.detach().numpy().transpose(0, 2, 1, 3), atol=1e-12)
    np.testing.assert_allclose(dq, tq.grad.numpy().transpose(0, 2, 1, 3), atol=1e-11)
    np.testing.assert_allclose(dk, tk.grad.numpy().transpose(0, 2, 1, 3), atol=1e-11)
    np.testing.assert_allclose(dv, tv.grad.numpy().transpose(0, 2, 1, 3), atol=1e-11)
    np.testing.assert_allclose(db, tb.grad.numpy(), atol=1e-11)


def test_central_finite_differences(rng):
    """Gradients of L = sum(dO * O) w.r.t. Q, K, V and bias by central
    differences (h = 1e-6), with segments, padding, GQA and causal masking."""
    B, S, Hq, Hkv, Dk, Dv = 1, 6, 2, 1, 3, 2
    q, k, v, do = rand(rng, B, S, Hq, Dk), rand(rng, B, S, Hkv, Dk), rand(rng, B, S, Hkv, Dv), rand(
        rng, B, S, Hq, Dv)
    ids, pos = seg_meta([[2, 3]], S)
    bias = 0.5 * rand(rng, 1, Hq, S, S)
    scale = 0.8

    def loss(q_, k_, v_, b_):
        o, _ = R.attention_forward(q_, k_, v_, ids, pos, ids, pos, True, scale, b_)
        return float((do * o).sum())

    grads = R.attention_backward(q, k, v, do, ids, pos, ids, pos, True, scale, bias)
    h = 1e-6
    for which, (arr, g) in enumerate(zip((q, k, v, bias), grads)):
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            args = [q.copy(), k.copy(), v.copy(), bias.copy()]
            args[which][idx] += h
            lp = loss(*args)
            args[which][idx] -= 2 * h
            lm = loss(*args)
            fd[idx] = (lp - lm) / (2 * h)
        err = np.abs(fd - g).max() / max(np.abs(g).max(), 1e-30)
        assert err <= 1e-6, (which, err)


def test_softmax_rows_sum_to_one(rng):
    """With V = 1 every valid output row is exactly the softmax row sum (= 1)."""
    prob = list(small_problem(rng, cross=True, Skv=12, with_bias=True))
    prob[2] = np.ones_like(prob[2])
    q, k, v, do, idq, posq, idk, posk, causal, scale, bias = prob
    o, lse = R.attention_forward(q, k, v, idq, posq, idk, posk, causal, scale, bias)
    has = np.isfinite(lse).transpose(0, 2, 1)  # [B,S,H]
    assert np.abs(o[has] - 1.0).max() <= 1e-12
    assert np.all(o[~has] == 0.0)


def test_closed_form_two_keys():
    """One head, d=1: Q=[1,2], K=[1,0], V=[1,3], scale 1, causal.
    Row 0 sees key 0 only: O=1, LSE=1.  Row 1: weights e^2 and 1."""
    q = np.array([1.0, 2.0]).reshape(1, 2, 1, 1)
    k = np.array([1.0, 0.0]).reshape(1, 2, 1, 1)
    v = np.array([1.0, 3.0]).reshape(1, 2, 1, 1)
    ids, pos = R.dense_metadata(1, 2)
    o, lse = R.attention_forward(q, k, v, ids, pos, ids, pos, True, 1.0)
    e2 = math.exp(2.0)
    assert o[0, 0, 0, 0] == pytest.approx(1.0, abs=1e-15)
    assert lse[0, 0, 0] == pytest.approx(1.0, abs=1e-15)
    assert o[0, 1, 0, 0] == pytest.approx((e2 + 3.0) / (e2 + 1.0), abs=1e-15)
    assert lse[0, 0, 1] == pytest.approx(math.log(e2 + 1.0), abs=1e-15)
    # dO = 1 on row 1 only: dV_1 = P_11 = 1/(e^2+1); dV_0 gets 1 (row 0) * 0 + P_10.
    do = np.array([0.0, 1.0]).reshape(1, 2, 1, 1)
    _, _, dv, _ = R.attention_backward(q, k, v, do, ids, pos, ids, pos, True, 1.0)
    assert dv[0, 1, 0, 0] == pytest.approx(1.0 / (e2 + 1.0), abs=1e-15)
    assert dv[0, 0, 0, 0] == pytest.approx(e2 / (e2 + 1.0), abs=1e-15)


def test_dv_is_pt_do_and_D_identity(rng):
    """dV = P^T dO with P formed explicitly, and rowsum(dO*O) = rowsum(P*dP)."""
    B, S, H, D = 1, 10, 1, 4
    q, k, v, do = rand(rng, B, S, H, D), rand(rng, B, S, H, D), rand(rng, B, S, H, D), rand(
        rng, B, S, H, D)
    ids, pos = seg_meta([[6, 3]], S)
    o, lse = R.attention_forward(q, k, v, ids, pos, ids, pos, True, 0.5)
    _, _, dv, _ = R.attention_backward(q, k, v, do, ids, pos, ids, pos, True, 0.5)
    mask = R.valid_pairs(ids[0], pos[0], ids[0], pos[0], True)
    s = 0.5 * q[0, :, 0] @ k[0, :, 0].T
    P = np.where(mask, np.exp(s - np.where(np.isfinite(lse[0, 0]), lse[0, 0], 0)[:, None]), 0.0)
    np.testing.assert_allclose(dv[0, :, 0], P.T @ do[0, :, 0], atol=1e-12)
    dP = do[0, :, 0] @ v[0, :, 0].T
    np.testing.assert_allclose((do[0, :, 0] * o[0, :, 0]).sum(1), (P * dP).sum(1), atol=1e-12)


def test_fully_masked_rows_give_zero(rng):
    """Query ids with no KV counterpart and padding rows: O = 0, LSE = -inf,
    dQ = 0, and they contribute nothing to dK/dV."""
    B, S, H, D = 1, 8, 2, 4
    q, k, v, do = rand(rng, B, S, H, D), rand(rng, B, S, H, D), rand(rng, B, S, H, D), rand(
        rng, B, S, H, D)
    idq = np.array([[1, 1, 3, 3, 2, 2, 0, 0]])
    idk = np.array([[1, 1, 1, 2, 2, 2, 0, 0]])
    pq, pk = R.derive_segment_pos(idq), R.derive_segment_pos(idk)
    o, lse = R.attention_forward(q, k, v, idq, pq, idk, pk, False, 0.5)
    dq, dk, dv, _ = R.attention_backward(q, k, v, do, idq, pq, idk, pk, False, 0.5)
    dead = [2, 3, 6, 7]
    assert np.all(o[0, dead] == 0) and np.all(dq[0, dead] == 0)
    assert np.all(np.isneginf(lse[0][:, dead]))
    assert np.all(dk[0, 6:] == 0) and np.all(dv[0, 6:] == 0)
    # changing the dead rows' Q and dO changes nothing else
    q2, do2 = q.copy(), do.copy()
    q2[0, dead] = 1000.0
    do2[0, dead] = -7.0
    _, dk2, dv2, _ = R.attention_backward(q2, k, v, do2, idq, pq, idk, pk, False, 0.5)
    assert np.array_equal(dk, dk2) and np.array_equal(dv, dv2)


def test_empty_segment_and_one_sided_id(rng):
    """A duplicated ragged offset (empty segment) changes nothing; a KV-only
    segment id leaves every query output unchanged and gets zero dK/dV."""
    T, H, D = 9, 2, 4
    q, k, v, do = rand(rng, 1, T, H, D), rand(rng, 1, T, H, D), rand(rng, 1, T, H, D), rand(
        rng, 1, T, H, D)
    a = R.metadata_from_cu_seqlens([0, 3, 7], T)
    b = R.metadata_from_cu_seqlens([0, 3, 3, 7], T)
    # the empty segment shifts later ids by one on both sides alike
    ra = run_oracle(R, (q, k, v, do, a[0], a[1], a[0], a[1], True, 0.6, None))
    rb = run_oracle(R, (q, k, v, do, b[0], b[1], b[0], b[1], True, 0.6, None))
    for x, y in zip(ra, rb):
        assert_same(x, y, tol=0)
    # KV side: tokens 7,8 become a segment with an id absent from Q
    idk = a[0].copy()
    idk[0, 7:] = 5
    pk = R.derive_segment_pos(idk)
    rc = run_oracle(R, (q, k, v, do, a[0], a[1], idk, pk, True, 0.6, None))
    for x, y in zip(ra[:3], rc[:3]):
        assert_same(x, y, tol=0)
    assert np.all(rc[3][0, 7:] == 0) and np.all(rc[4][0, 7:] == 0)


def test_segment_permutation_equivariance(rng):
    """Permuting whole segments inside a packed row (positions restart) permutes
    O/LSE/dQ/dK/dV the same way, under a nonuniform dO."""
    lens = [3, 5, 4]
    S = 14  # 2 padding tokens
    q, k, v, do = rand(rng, 1, S, 4, 3), rand(rng, 1, S, 2, 3), rand(rng, 1, S, 2, 5), rand(
        rng, 1, S, 4, 5)
    ids, pos = seg_meta([lens], S)
    starts = np.cumsum([0] + lens)
    order = [2, 0, 1]
    perm = np.concatenate([np.arange(starts[s], starts[s] + lens[s]) for s in order] +
                          [np.arange(12, 14)])
    ids_p, pos_p = seg_meta([[lens[s] for s in order]], S)
    r1 = run_oracle(R, (q, k, v, do, ids, pos, ids, pos, True, 0.5, None))
    r2 = run_oracle(R, (q[:, perm], k[:, perm], v[:, perm], do[:, perm], ids_p, pos_p, ids_p,
                        pos_p, True, 0.5, None))
    np.testing.assert_allclose(r2[0], r1[0][:, perm], atol=1e-13)
    assert_same(r2[1], r1[1][:, :, perm], tol=1e-13)
    for t in (2, 3, 4):
        np.testing.assert_allclose(r2[t], r1[t][:, perm], atol=1e-13)


def test_packing_equals_separate_dense_causal(rng):
    """A packed row equals each segment run alone as dense causal attention
    (torch SDPA in float64)."""
    lens = [4, 6, 3]
    S = sum(lens) + 2
    H, D = 2, 5
    q, k, v = rand(rng, 1, S, H, D), rand(rng, 1, S, H, D), rand(rng, 1, S, H, D)
    ids, pos = seg_meta([lens], S)
    o, _ = R.attention_forward(q, k, v, ids, pos, ids, pos, True, 0.3)
    t = 0
    for L in lens:
        sl = slice(t, t + L)
        ref = torch.nn.functional.scaled_dot_product_attention(
            *(torch.tensor(x[0, sl].transpose(1, 0, 2)) for x in (q, k, v)), is_causal=True,
            scale=0.3)
        np.testing.assert_allclose(o[0, sl], ref.numpy().transpose(1, 0, 2), atol=1e-13)
        t += L


def test_gqa_equals_repeated_heads(rng):
    B, S, Hq, Hkv, D = 1, 9, 6, 2, 4
    q, k, v, do = rand(rng, B, S, Hq, D), rand(rng, B, S, Hkv, D), rand(rng, B, S, Hkv, D), rand(
        rng, B, S, Hq, D)
    ids, pos = seg_meta([[5, 3]], S)
    r = run_oracle(R, (q, k, v, do, ids, pos, ids, pos, True, 0.5, None))
    ke, ve = np.repeat(k, Hq // Hkv, axis=2), np.repeat(v, Hq // Hkv, axis=2)
    re = run_oracle(R, (q, ke, ve, do, ids, pos, ids, pos, True, 0.5, None))
    np.testing.assert_allclose(r[0], re[0], atol=1e-13)
    np.testing.assert_allclose(r[2], re[2], atol=1e-13)
    np.testing.assert_allclose(r[3], re[3].reshape(B, S, Hkv, Hq // Hkv, D).sum(3), atol=1e-13)
    np.testing.assert_allclose(r[4], re[4].reshape(B, S, Hkv, Hq // Hkv, D).sum(3), atol=1e-13)


def test_sampled_evaluation_matches_full(rng):
    prob = small_problem(rng, cross=True, Skv=12, bias_shape=(1, 4, 11, 12))
    q, k, v, do, idq, posq, idk, posk, causal, scale, bias = prob
    o, lse, dq, dk, dv, _ = run_oracle(R, prob)
    rows = [0, 3, 8, 10]
    for b in range(2):
        for h in range(4):
            so, sl = R.forward_rows(q, k, v, idq, posq, idk, posk, causal, scale, b, h, rows, bias)
            np.testing.assert_allclose(so, o[b, rows, h], atol=1e-13)
            assert_same(sl, lse[b, h, rows], tol=1e-13)
            sd = R.backward_dq_rows(q, k, v, do, idq, posq, idk, posk, causal, scale, b, h, rows,
                                    bias)
            np.testing.assert_allclose(sd, dq[b, rows, h], atol=1e-13)
        for g in range(2):
            cols = [0, 5, 11]
            sk, sv = R.backward_dkdv_cols(q, k, v, do, idq, posq, idk, posk, causal, scale, b, g,
                                          cols, bias)
            np.testing.assert_allclose(sk, dk[b, cols, g], atol=1e-13)
            np.testing.assert_allclose(sv, dv[b, cols, g], atol=1e-13)


# ----------------------------------------------------------------- metadata / layouts


def test_derive_segment_pos_and_cu_seqlens():
    ids = np.array([[1, 1, 1, 2, 2, 0, 0], [3, 3, 1, 1, 1, 1, 0]])
    np.testing.assert_array_equal(R.derive_segment_pos(ids),
                                  [[0, 1, 2, 0, 1, 0, 1], [0, 1, 0, 1, 2, 3, 0]])
    i, p = R.metadata_from_cu_seqlens([0, 2, 5], 7)
    np.testing.assert_array_equal(i, [[1, 1, 2, 2, 2, 0, 0]])
    np.testing.assert_array_equal(p[0, :5], [0, 1, 0, 1, 2])


def test_layout_3hd_reduces_to_T3HD(rng):
    """With Hq == Hkv and d_qk == d_v the generalised 3HD packing is the
    [T, 3, H, D] packing: K one head-block and V two head-blocks after Q."""
    B, S, H, D = 2, 5, 3, 4
    buf = rand(rng, B * S, 3, H, D)
    q, k, v = R.unpack_layout("3HD", {"qkv": buf.reshape(B * S, -1)}, B, S, S, H, H, D, D)
    np.testing.assert_array_equal(q.reshape(B * S, H, D), buf[:, 0])
    np.testing.assert_array_equal(k.reshape(B * S, H, D), buf[:, 1])
    np.testing.assert_array_equal(v.reshape(B * S, H, D), buf[:, 2])


def test_layout_offsets_golden():
    """Element offsets of the K/V slices against the fixture derived from the
    page's pointer arithmetic (stride = typeSize * heads * head_dim)."""
    import json
    import os

    with open(os.path.join(os.path.dirname(__file__), "golden", "layout_offsets.json")) as f:
        gold = json.load(f)
    for c in gold["cases"]:
        Hq, Hkv, dqk, dv = c["Hq"], c["Hkv"], c["d_qk"], c["d_v"]
        T = 2
        if c["layout"] == "3HD":
            W = Hq * dqk + Hkv * dqk + Hkv * dv
            buf = np.arange(T * W, dtype=np.float64).reshape(T, W)
            q, k, v = R.unpack_layout("3HD", {"qkv": buf}, 1, T, T, Hq, Hkv, dqk, dv)
            assert k[0, 0, 0, 0] * 2 == c["k_offset_bytes"]
            assert v[0, 0, 0, 0] * 2 == c["v_offset_bytes"]
            assert (q[0, 1, 0, 0] - q[0, 0, 0, 0]) * 2 == c["token_stride_bytes"]
        else:
            buf = np.arange(T * 2 * Hkv * dv, dtype=np.float64).reshape(T, 2, Hkv, dv)
            _, k, v = R.unpack_layout("HD_2HD", {"q": np.zeros((T, Hq * dqk)), "kv": buf}, 1, T,
                                      T, Hq, Hkv, dqk, dv)
            assert (v[0, 0, 0, 0] - k[0, 0, 0, 0]) * 2 == c["v_offset_bytes"]
            assert (k[0, 1, 0, 0] - k[0, 0, 0, 0]) * 2 == c["token_stride_bytes"]


def test_layout_checks():
    with pytest.raises(ValueError):
        R.unpack_layout("3HD", {"qkv": np.zeros((4, 24))}, 1, 4, 5, 2, 2, 4, 4)
    with pytest.raises(ValueError):
        R.unpack_layout("HD_2HD", {"q": np.zeros((4, 8)), "kv": np.zeros((4, 2, 2, 2))}, 1, 4, 4,
                        2, 2, 4, 2)


# ----------------------------------------------------------------- band masks


@pytest.mark.parametrize("band", [(3, 0, 0), (2, 1, 0), (None, 0, 2), (1, None, -1)])
def test_window_brute_force(rng, band):
    """Sliding windows, a two-sided band and shifted alignments against the
    scalar loops (which test the band condition on their own)."""
    prob = small_problem(rng, S=11, bias_shape=(1, 4, 11, 11))
    q, k, v, do, idq, posq, idk, posk, _, scale, bias = prob
    w = R.Window(*band)
    o, lse = R.attention_forward(q, k, v, idq, posq, idk, posk, w, scale, bias, row_block=4)
    g = R.attention_backward(q, k, v, do, idq, posq, idk, posk, w, scale, bias, row_block=4)
    ref = brute_force(q, k, v, do, idq, posq, idk, posk, band, scale, bias)
    for a, b in zip((o, lse) + tuple(g), ref):
        assert_same(a, b, tol=1e-10)


def test_window_limits_and_closed_forms(rng):
    """Window(None, 0) is the causal mask and Window(None, None) no mask; a
    zero-width window keeps only the diagonal, so O_i = V_i and LSE_i = S_ii;
    bottom-right alignment of dense rows: the last query row sees every key."""
    prob = small_problem(rng, S=11, with_bias=False)
    q, k, v, do, idq, posq, idk, posk, _, scale, _ = prob
    for w, flag in ((R.Window(None, 0), True), (R.Window(None, None), False)):
        a = R.attention_forward(q, k, v, idq, posq, idk, posk, w, scale)
        b = R.attention_forward(q, k, v, idq, posq, idk, posk, flag, scale)
        for x, y in zip(a, b):
            assert_same(x, y, tol=1e-13)
    B, S, Hq, Hkv, D = 1, 6, 2, 2, 4
    q, k, v = rand(rng, B, S, Hq, D), rand(rng, B, S, Hkv, D), rand(rng, B, S, Hkv, 3)
    ids, pos = R.dense_metadata(B, S)
    o, lse = R.attention_forward(q, k, v, ids, pos, ids, pos, R.Window(0, 0), 0.5)
    np.testing.assert_allclose(o[0], v[0], atol=1e-13)
    np.testing.assert_allclose(lse[0], 0.5 * np.einsum("shd,shd->hs", q[0], k[0]), atol=1e-13)
    Sq, Skv = 3, 7
    q, k, v = rand(rng, 1, Sq, 1, D), rand(rng, 1, Skv, 1, D), rand(rng, 1, Skv, 1, 3)
    iq, pq = R.dense_metadata(1, Sq)
    ik, pk = R.dense_metadata(1, Skv)
    _, lse = R.attention_forward(q, k, v, iq, pq, ik, pk, R.Window(None, 0, Skv - Sq), 0.5)
    s_last = 0.5 * k[0, :, 0] @ q[0, -1, 0]
    assert abs(lse[0, 0, -1] - (s_last.max() + np.log(np.exp(s_last - s_last.max()).sum()))) < 1e-12
    assert R.count_valid_pairs(iq, pq, ik, pk, R.Window(None, 0, Skv - Sq)) == 5 + 6 + 7


# ----------------------------------------------------------------- sink attention


@pytest.mark.parametrize("cross", [False, True])
def test_sink_brute_force(rng, cross):
    prob = small_problem(rng, S=9, Skv=12 if cross else None, cross=cross,
                         bias_shape=(1, 4, 9, 12 if cross else 9))
    q, k, v, do, idq, posq, idk, posk, causal, scale, bias = prob
    sink = rng.standard_normal(q.shape[2]) * 2.0
    o, lse = R.attention_forward(q, k, v, idq, posq, idk, posk, causal, scale, bias,
                                 row_block=4, sink=sink)
    dq, dk, dv, db = R.attention_backward(q, k, v, do, idq, posq, idk, posk, causal, scale,
                                          bias, row_block=4, sink=sink)
    ref = brute_force(q, k, v, do, idq, posq, idk, posk, causal, scale, bias, sink=sink)
    for a, b in zip((o, lse, dq, dk, dv, db), ref):
        assert_same(a, b, tol=1e-10)
    # rows without valid keys: O = 0 and LSE = the sink
    assert np.all(np.isfinite(lse))


def test_sink_minus_infinity_is_no_sink(rng):
    prob = small_problem(rng, S=9)
    q, k, v, do, idq, posq, idk, posk, causal, scale, bias = prob
    none = run_oracle(R, prob)
    sink = np.full(q.shape[2], -np.inf)
    o, lse = R.attention_forward(q, k, v, idq, posq, idk, posk, causal, scale, bias, sink=sink)
    g = R.attention_backward(q, k, v, do, idq, posq, idk, posk, causal, scale, bias, sink=sink)
    for a, b in zip((o, lse) + tuple(g), none):
        assert_same(a, b, tol=1e-13)


def test_sink_gradient_finite_differences_and_row_sums(rng):
    """dsink against central differences of L = sum(dO * O); each row's key
    probabilities plus the sink's sum to 1."""
    prob = small_problem(rng, S=11, bias_shape=(1, 4, 11, 11))
    q, k, v, do, idq, posq, idk, posk, causal, scale, bias = prob
    sink = rng.standard_normal(q.shape[2])
    ds = R.sink_gradient(q, k, v, do, idq, posq, idk, posk, causal, scale, sink, bias,
                         row_block=3)

    def loss(sk):
        o, _ = R.attention_forward(q, k, v, idq, posq, idk, posk, causal, scale, bias, sink=sk)
        return float((do * o).sum())

    eps = 1e-6
    for h in range(q.shape[2]):
        sp, sm = sink.copy(), sink.copy()
        sp[h] += eps
        sm[h] -= eps
        fd = (loss(sp) - loss(sm)) / (2 * eps)
        assert abs(fd - ds[h]) <= 1e-6 * max(1.0, abs(fd)), (h, fd, ds[h])
    b, h = 0, 1
    mask = R.valid_pairs(idq[b], posq[b], idk[b], posk[b], causal)
    cols, _, p, m, l = R._rows_softmax(q[b, :, h], k[b, :, h // 2], mask, scale,
                                       bias[0, h], float(sink[h]))
    has = mask.any(axis=1)
    total = p.sum(axis=1) + np.exp(sink[h] - m) / l
    np.testing.assert_allclose(total[has], 1.0, atol=1e-13)


# ----------------------------------------------------------------- max-logit


def brute_max_logit(q, k, idq, posq, idk, posk, causal, scale, bias=None):
    """Pure-Python loops: largest valid S_ij per (b, h)."""
    B, Sq, Hq, Dk = q.shape
    Skv, Hkv = k.shape[1], k.shape[2]
    out = np.full((B, Hq), -np.inf)
    for b in range(B):
        for h in range(Hq):
            g = h // (Hq // Hkv)
            bb = b if (bias is not None and bias.shape[0] > 1) else 0
            bh = h if (bias is not None and bias.shape[1] > 1) else 0
            for i in range(Sq):
                for j in range(Skv):
                    ok = idq[b, i] == idk[b, j] and idq[b, i] != 0
                    if causal:
                        ok = ok and posk[b, j] <= posq[b, i]
                    if not ok:
                        continue
                    acc = sum(q[b, i, h, c] * k[b, j, g, c] for c in range(Dk)) * scale
                    if bias is not None:
                        acc += bias[bb, bh, i, j]
                    out[b, h] = max(out[b, h], acc)
    return out


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("cross", [False, True])
def test_max_logit_brute_force(rng, causal, cross):
    q, k, v, do, idq, posq, idk, posk, causal, scale, bias = small_problem(
        rng, causal=causal, cross=cross, S=9, Skv=12 if cross else None,
        bias_shape=(2, 1, 9, 12 if cross else 9))
    got = R.max_logit(q, k, idq, posq, idk, posk, causal, scale, bias, row_block=4)
    ref = brute_max_logit(q, k, idq, posq, idk, posk, causal, scale, bias)
    assert_same(got, ref, tol=1e-12)


def test_max_logit_single_key_rows_and_lse_bounds(rng):
    """With one valid key per row, LSE_i is that key's logit, so the max-logit
    is the largest LSE; in general max_i (LSE_i - ln n_i) <= max-logit <=
    max_i LSE_i, n_i the row's number of valid keys (the forward's LSE)."""
    B, S, Hq, Hkv, D = 2, 7, 4, 2, 5
    q, k = rand(rng, B, S, Hq, D), rand(rng, B, S, Hkv, D)
    v = rand(rng, B, S, Hkv, 3)
    ids, pos = seg_meta([[1] * 6, [1] * 4], S)  # segments of one token, then padding
    ml = R.max_logit(q, k, ids, pos, ids, pos, True, 0.8)
    _, lse = R.attention_forward(q, k, v, ids, pos, ids, pos, True, 0.8)
    np.testing.assert_allclose(ml, lse.max(axis=2), rtol=0, atol=1e-12)
    q, k, v, do, idq, posq, idk, posk, causal, scale, bias = small_problem(rng, cross=True,
                                                                           Skv=13)
    ml = R.max_logit(q, k, idq, posq, idk, posk, causal, scale, bias)
    _, lse = R.attention_forward(q, k, v, idq, posq, idk, posk, causal, scale, bias)
    for b in range(q.shape[0]):
        n = R.valid_pairs(idq[b], posq[b], idk[b], posk[b], causal).sum(axis=1)
        has = n > 0
        for h in range(q.shape[2]):
            lo = np.max(lse[b, h, has] - np.log(n[has]))
            hi = np.max(lse[b, h, has])
            assert lo - 1e-12 <= ml[b, h] <= hi + 1e-12


def test_max_logit_planted_mistake_caught(rng):
    """Keeping only the last row block's maximum disagrees with the loops."""
    prob = small_problem(rng, S=11, bias_shape=(1, 4, 11, 11))
    q, k, v, do, idq, posq, idk, posk, causal, scale, bias = prob
    ref = brute_max_logit(q, k, idq, posq, idk, posk, causal, scale, bias)
    bad = _mutant("out[b, h] = max(out[b, h], float(m.max()))", "out[b, h] = float(m.max())")
    got = bad.max_logit(q, k, idq, posq, idk, posk, causal, scale, bias, row_block=4)
    assert not np.allclose(got, ref)


# ----------------------------------------------------------------- planted mistakes

MUTATIONS = [
    ("ds = p * (dp - D[:, None])", "ds = p * (dp + D[:, None])"),  # wrong sign
    ("dq[b, r0:r1, h] = scale * (ds @", "dq[b, r0:r1, h] = (ds @"),  # dropped factor
    ("g = h // group", "g = h % Hkv"),  # wrong GQA head mapping
    ("dv[b, cols, g] += p.T @ do_r", "dv[b, cols, g] += p.T @ do_r[::-1]"),  # misplaced rows
    ("m &= np.asarray(pos_kv)[None, :] <= np.asarray(pos_q)[:, None]",
     "m &= np.asarray(pos_kv)[None, :] < np.asarray(pos_q)[:, None]"),  # off-by-one causal
    ("s = s + bias_rows[:, cols]", "s = s + bias_rows[::-1][:, cols]"),  # bias rows misplaced
    ("dbias[bi, hi, r0:r1][:, cols] += ds", "dbias[bi, hi, r0:r1][:, cols] = ds"),  # no reduction
    ("lse[b, h, r0:r1][fin] = m[fin] + np.log(l[fin])", "lse[b, h, r0:r1][fin] = m[fin]"),
]


def _mutant(old, new):
    import inspect

    src = inspect.getsource(R)
    assert src.count(old) >= 1, old
    mod = types.ModuleType("oracle_mutant")
    exec(compile(src.replace(old, new, 1), "oracle_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("old,new", MUTATIONS)
def test_pins_catch_planted_mistake(old, new):
    """Every planted mistake makes the oracle disagree with the brute-force pin
    on a problem with segments, GQA, causal masking and a broadcast bias."""
    rng = np.random.default_rng(7)
    prob = small_problem(rng, bias_shape=(1, 4, 11, 11), S=11)
    ref = brute_force(*prob)
    got = run_oracle(_mutant(old, new), prob)
    caught = False
    for a, b in zip(got, ref):
        try:
            assert_same(a, b)
        except AssertionError:
            caught = True
    assert caught, f"mutation not caught: {new}"


@pytest.mark.parametrize("old,new", [
    ("out[h] -= float((p_sink * D).sum())", "out[h] += float((p_sink * D).sum())"),
    ("l[finite] += np.exp(sink - m[finite])", "l[finite] += 0.0"),
    ("m = np.maximum(m, sink)", "m = m"),
])
def test_sink_pins_catch_planted_mistake(old, new):
    """A flipped sink-gradient sign, a normaliser without the sink, or a max
    that ignores the sink each disagree with the loops or the differences."""
    rng = np.random.default_rng(11)
    prob = small_problem(rng, S=11, bias_shape=(1, 4, 11, 11))
    q, k, v, do, idq, posq, idk, posk, causal, scale, bias = prob
    sink = rng.standard_normal(q.shape[2]) + 3.0  # above most logits
    bad = _mutant(old, new)
    ref = brute_force(q, k, v, do, idq, posq, idk, posk, causal, scale, bias, sink=sink)
    with np.errstate(all="ignore"):  # a mutant may divide by zero
        o, lse = bad.attention_forward(q, k, v, idq, posq, idk, posk, causal, scale, bias,
                                       sink=sink)
        ds = bad.sink_gradient(q, k, v, do, idq, posq, idk, posk, causal, scale, sink, bias)
    fwd_ok = np.allclose(o, ref[0], atol=1e-10) and np.allclose(lse, ref[1], atol=1e-10)

    def loss(sk):
        o2, _ = R.attention_forward(q, k, v, idq, posq, idk, posk, causal, scale, bias, sink=sk)
        return float((do * o2).sum())

    eps = 1e-6
    fd = []
    for h in range(q.shape[2]):
        sp, sm = sink.copy(), sink.copy()
        sp[h] += eps
        sm[h] -= eps
        fd.append((loss(sp) - loss(sm)) / (2 * eps))
    grad_ok = np.allclose(ds, fd, atol=1e-6)
    assert not (fwd_ok and grad_ok), f"mutation not caught: {new}"


@pytest.mark.parametrize("old,new", [
    ("m &= r >= -self.left", "m &= r > -self.left"),  # window one key short
    ("r = np.asarray(pos_kv)[None, :] - (np.asarray(pos_q)[:, None] + self.shift)",
     "r = np.asarray(pos_kv)[None, :] - (np.asarray(pos_q)[:, None] - self.shift)"),  # shift sign
])
def test_window_pins_catch_planted_mistake(old, new):
    rng = np.random.default_rng(5)
    prob = small_problem(rng, S=11, bias_shape=(1, 4, 11, 11))
    q, k, v, do, idq, posq, idk, posk, _, scale, bias = prob
    band = (3, 0, 1)
    bad = _mutant(old, new)
    o, lse = bad.attention_forward(q, k, v, idq, posq, idk, posk, bad.Window(*band), scale, bias)
    ref = brute_force(q, k, v, do, idq, posq, idk, posk, band, scale, bias)
    same = True
    for a, b in zip((o, lse), ref[:2]):
        try:
            assert_same(a, b)
        except AssertionError:
            same = False
    assert not same, f"mutation not caught: {new}"
