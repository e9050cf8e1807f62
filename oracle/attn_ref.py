"""Float64 CPU oracle for fused scaled-dot-product attention, forward and backward.

TEST INFRASTRUCTURE ONLY.  This module is the correctness reference for the
CUDA library in ``bwd_tcgen05_tma_gb300``.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline / reference arm of
``bench.py`` may import it.  The product path never calls it, and it shares no
code, helper, table or constant with the CUDA path.

What it computes (all in float64 on bf16-valued inputs):

* Layout resolution: the packed-QKV ("3HD"), packed-KV ("HD_2HD") and separate
  ("HD_HD_HD") layouts, where the K and V slices of a packed buffer start one
  and two head-blocks after Q, and the V slice of a packed KV buffer is offset
  by ``num_gqa_groups * v_head_dim`` elements (TransformerEngine PR #2358 "[JAX]
  Make all jax attention calls use non-packed common calls": the pointer
  arithmetic sequence diagram and the review of the KV-packed stride).
* Segment metadata: segment ids with 0 meaning padding, segment positions that
  restart in each segment and may be derived from the ids
  (TransformerEngine PR #2692 "[JAX] Fix batcher in FusedAttn primitive for
  when seg ids bdims != seg pos bdims", Description), or ragged offsets
  (cu_seqlens).
* The attention itself, as the plain definition.  For batch b, query head h
  with KV head g = h // (Hq // Hkv), query i and key j::

      valid(i, j) = id_q[i] == id_kv[j] != 0  and (not causal or pos_kv[j] <= pos_q[i])
      S_ij   = scale * <Q_i, K_j> + bias_ij          over valid pairs, -inf elsewhere
      P_ij   = exp(S_ij - m_i) / l_i,  m_i = max_j S_ij,  l_i = sum_j exp(S_ij - m_i)
      O_i    = sum_j P_ij V_j,  LSE_i = m_i + ln l_i    (O_i = 0, LSE_i = -inf if no valid j)

  and the closed-form backward for a given dO::

      dP_ij = <dO_i, V_j>,  D_i = sum_j P_ij dP_ij,  dS_ij = P_ij (dP_ij - D_i)
      dQ_i  = scale * sum_j dS_ij K_j
      dK_j  = scale * sum_{h in group(g)} sum_i dS_ij Q_i
      dV_j  = sum_{h in group(g)} sum_i P_ij dO_i
      dBias = dS summed over every axis the bias is broadcast along

  The outputs and gradient set follow the fused-attention backward diagram of
  TransformerEngine PR #3516 "[JAX] Align fused attn backward output gradient
  sharding and other test strengthening" (saved O plus incoming dO give the
  Q/K/V and optional bias gradients); Q and KV metadata may differ (same page,
  Changes 3-4); gradients of a KV head sum over the query heads that share it
  (maxdiffusion PR #485, Summary: dK/dV held across Q blocks and GQA heads);
  the bias gradient is reduced over its broadcast axes (PR #3516, Change 6).
* Optionally the max-logit output: per batch row and query head, the largest
  S_ij over valid pairs (``max_logit``; reading stated there).
* Optionally a band mask (``Window``: sliding windows, bottom-right causal
  alignment) in place of the causal flag; reading stated there.
* Optionally per-head sink logits that join every softmax row as a column
  without a value vector, and their gradient (``attention_forward``,
  ``sink_gradient``; reading stated there).
* An FP8 forward (``attention_forward_fp8``): Q, K, V given as E4M3 values with
  one descale factor per tensor, P quantised to E4M3 before it meets V
  (``e4m3_round``); reading stated there.

Rows are processed one block of queries at a time and each block only touches
the keys that are valid for at least one of its rows; since every softmax row is
independent and masked keys contribute exactly zero, this is still the plain
definition, not a reformulation.
"""
from __future__ import annotations

import numpy as np

LAYOUTS = ("3HD", "HD_2HD", "HD_HD_HD")

# --------------------------------------------------------------------------
# Layout resolution
# --------------------------------------------------------------------------


def unpack_layout(layout, buffers, B, Sq, Skv, Hq, Hkv, d_qk, d_v):
    """Return float64 views Q [B,Sq,Hq,d_qk], K [B,Skv,Hkv,d_qk], V [B,Skv,Hkv,d_v].

    ``buffers`` holds the raw token-major arrays of the layout:

    * "3HD":      {"qkv": [B*Sq, Hq*d_qk + Hkv*d_qk + Hkv*d_v]} -- each token row
      packs the Q heads, then the K heads, then the V heads.  With Hq == Hkv and
      d_qk == d_v this is the [T, 3, H, D] packing with K one head-block and V
      two head-blocks after Q (PR #2358, pointer arithmetic for NVTE_3HD).
      Requires Sq == Skv (PR #2358, the q_max_seqlen == kv_max_seqlen check).
    * "HD_2HD":   {"q": [B*Sq, Hq*d_qk], "kv": [B*Skv, 2, Hkv, d_v]} -- the V
      slice starts Hkv*d_v elements after the K slice (PR #2358, KV-packed stride
      review); requires d_qk == d_v.
    * "HD_HD_HD": {"q": ..., "k": ..., "v": ...} separate arrays.
    """
    if layout == "3HD":
        if Sq != Skv:
            raise ValueError("3HD needs equal query and key/value lengths")
        qkv = np.asarray(buffers["qkv"], dtype=np.float64).reshape(B * Sq, -1)
        if qkv.shape[1] != Hq * d_qk + Hkv * d_qk + Hkv * d_v:
            raise ValueError("3HD row width mismatch")
        q = qkv[:, : Hq * d_qk]
        k = qkv[:, Hq * d_qk : Hq * d_qk + Hkv * d_qk]
        v = qkv[:, Hq * d_qk + Hkv * d_qk :]
    elif layout == "HD_2HD":
        if d_qk != d_v:
            raise ValueError("HD_2HD needs qk_head_dim == v_head_dim")
        q = np.asarray(buffers["q"], dtype=np.float64).reshape(B * Sq, -1)
        kv = np.asarray(buffers["kv"], dtype=np.float64).reshape(B * Skv, 2 * Hkv * d_v)
        k = kv[:, : Hkv * d_v]
        v = kv[:, Hkv * d_v :]
    elif layout == "HD_HD_HD":
        q = np.asarray(buffers["q"], dtype=np.float64)
        k = np.asarray(buffers["k"], dtype=np.float64)
        v = np.asarray(buffers["v"], dtype=np.float64)
    else:
        raise ValueError(f"unknown layout {layout!r}")
    return (
        q.reshape(B, Sq, Hq, d_qk),
        k.reshape(B, Skv, Hkv, d_qk),
        v.reshape(B, Skv, Hkv, d_v),
    )


# --------------------------------------------------------------------------
# Segment metadata
# --------------------------------------------------------------------------


def derive_segment_pos(segment_ids):
    """Positions restarting at 0 at the first token of every run of equal ids
    (what from_segment_ids_and_pos generates when only ids are given, PR #2692,
    Description).  Works row by row on a [B, S] array."""
    ids = np.asarray(segment_ids)
    pos = np.zeros(ids.shape, dtype=np.int64)
    for b in range(ids.shape[0]):
        p = 0
        for t in range(ids.shape[1]):
            if t > 0 and ids[b, t] != ids[b, t - 1]:
                p = 0
            pos[b, t] = p
            p += 1
    return pos


def metadata_from_cu_seqlens(cu_seqlens, total):
    """Ragged offsets -> ([1, total] ids, [1, total] pos).  Segment k covers
    tokens cu[k] .. cu[k+1]-1 and gets id k+1; tokens at or past cu[n] are
    padding (id 0); equal consecutive offsets describe an empty segment."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    ids = np.zeros((1, total), dtype=np.int64)
    pos = np.zeros((1, total), dtype=np.int64)
    for k in range(len(cu) - 1):
        lo, hi = int(cu[k]), int(cu[k + 1])
        ids[0, lo:hi] = k + 1
        pos[0, lo:hi] = np.arange(hi - lo)
    return ids, pos


def dense_metadata(B, S):
    """Dense BSHD rows without segments: every token valid, position = index."""
    return np.ones((B, S), dtype=np.int64), np.tile(np.arange(S, dtype=np.int64), (B, 1))


class Window:
    """A band of key positions relative to each query position, usable
    wherever a ``causal`` flag is taken: key j is kept when

        -left <= pos_kv[j] - (pos_q[i] + shift) <= right

    (None: unbounded on that side).  Window(None, 0) is the causal mask;
    Window(w - 1, 0) a causal sliding window of w keys; ``shift`` = Skv - Sq
    aligns a causal mask bottom-right for dense rows of unequal lengths.

    The pages do not define windows or bottom-right alignment; this is the
    usual reading, kept here so the "next" mask variants have a pinned
    definition before any kernel implements them."""

    def __init__(self, left=None, right=0, shift=0):
        self.left, self.right, self.shift = left, right, shift

    def keep(self, pos_q, pos_kv):
        r = np.asarray(pos_kv)[None, :] - (np.asarray(pos_q)[:, None] + self.shift)
        m = np.ones(r.shape, dtype=bool)
        if self.left is not None:
            m &= r >= -self.left
        if self.right is not None:
            m &= r <= self.right
        return m


def valid_pairs(id_q, pos_q, id_kv, pos_kv, causal):
    """Boolean [Sq, Skv] mask of one batch row: same nonzero segment and, when
    causal, key position not after the query position (``causal`` may also
    be a Window)."""
    id_q = np.asarray(id_q)[:, None]
    id_kv = np.asarray(id_kv)[None, :]
    m = (id_q == id_kv) & (id_q != 0)
    if isinstance(causal, Window):
        m &= causal.keep(pos_q, pos_kv)
    elif causal:
        m &= np.asarray(pos_kv)[None, :] <= np.asarray(pos_q)[:, None]
    return m


def count_valid_pairs(id_q, pos_q, id_kv, pos_kv, causal):
    """Exact number of unmasked (i, j) pairs per head summed over batch rows."""
    return int(sum(valid_pairs(id_q[b], pos_q[b], id_kv[b], pos_kv[b], causal).sum()
                   for b in range(np.asarray(id_q).shape[0])))


# --------------------------------------------------------------------------
# The attention definition
# --------------------------------------------------------------------------


def _bias_index(bias_shape, b, h):
    bb, bh = bias_shape[0], bias_shape[1]
    return (b if bb > 1 else 0), (h if bh > 1 else 0)


def _rows_softmax(q_rows, k_b, mask_rows, scale, bias_rows, sink=None):
    """Scores and probabilities of a block of query rows over the keys valid
    for at least one of them.  Returns (cols, S, P, m, l).  With a sink logit
    (a float), every row's softmax runs over its valid logits and the sink:
    m and l include the sink, whose own probability is exp(sink - m) / l."""
    cols = np.nonzero(mask_rows.any(axis=0))[0]
    R = q_rows.shape[0]
    if cols.size == 0:
        if sink is not None and np.isfinite(sink):
            return cols, np.zeros((R, 0)), np.zeros((R, 0)), np.full(R, float(sink)), np.ones(R)
        return cols, np.zeros((R, 0)), np.zeros((R, 0)), np.full(R, -np.inf), np.zeros(R)
    s = scale * (q_rows @ k_b[cols].T)
    if bias_rows is not None:
        s = s + bias_rows[:, cols]
    s = np.where(mask_rows[:, cols], s, -np.inf)
    m = s.max(axis=1)
    if sink is not None:
        m = np.maximum(m, sink)
    finite = np.isfinite(m)
    e = np.zeros_like(s)
    e[finite] = np.exp(s[finite] - m[finite, None])
    l = e.sum(axis=1)
    if sink is not None:
        l[finite] += np.exp(sink - m[finite])
    p = np.zeros_like(e)
    p[finite] = e[finite] / l[finite, None]
    return cols, s, p, m, l


def attention_forward(q, k, v, id_q, pos_q, id_kv, pos_kv, causal, scale, bias=None,
                      row_block=256, sink=None):
    """O [B,Sq,Hq,d_v] and LSE [B,Hq,Sq] (natural log) by the definition above.

    sink: optional [Hq] per-head logits that join every row's softmax as one
    more column with no value vector (the sink attention of TransformerEngine
    PR #2225, which PR #2358 "[JAX] Make all jax attention calls use
    non-packed common calls" links without defining it; the reading is the
    usual one: the sink only enlarges the normaliser).  A row without valid
    keys then has O = 0 and LSE = sink."""
    B, Sq, Hq, _ = q.shape
    _, Skv, Hkv, d_v = v.shape
    group = Hq // Hkv
    o = np.zeros((B, Sq, Hq, d_v))
    lse = np.full((B, Hq, Sq), -np.inf)
    for b in range(B):
        mask = valid_pairs(id_q[b], pos_q[b], id_kv[b], pos_kv[b], causal)
        for h in range(Hq):
            g = h // group
            for r0 in range(0, Sq, row_block):
                r1 = min(Sq, r0 + row_block)
                br = None
                if bias is not None:
                    bi, hi = _bias_index(bias.shape, b, h)
                    br = bias[bi, hi, r0:r1]
                sk = None if sink is None else float(sink[h])
                cols, _, p, m, l = _rows_softmax(q[b, r0:r1, h], k[b, :, g], mask[r0:r1],
                                                 scale, br, sk)
                fin = np.isfinite(m)
                lse[b, h, r0:r1][fin] = m[fin] + np.log(l[fin])
                if cols.size == 0:
                    continue
                o[b, r0:r1, h] = p @ v[b, cols, g]
    return o, lse


# --------------------------------------------------------------------------
# FP8 (E4M3) forward
# --------------------------------------------------------------------------

E4M3_MAX = 448.0  # 1.75 * 2^8: the largest finite E4M3 value
P_SCALE = 256.0   # P is quantised as E4M3(256 * p), so p = 1 maps to 256


def e4m3_round(x):
    """Nearest E4M3 value (ties to even), saturating at +-448, from the format:
    1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; no infinities;
    normal values (1 + m/8) 2^e for e in [-6, 8] (the top code of e = 8 is
    NaN, so the largest is 1.75 * 2^8 = 448), subnormal values k 2^-9 for
    k = 0..7.  In every binade [2^e, 2^(e+1)) the spacing is 2^(e-3); below
    2^-6 it is 2^-9."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.clip(e, -6, 8)
    quantum = np.exp2(e - 3)  # 2^-9 in the subnormal range (e clamped to -6)
    r = np.rint(a / quantum) * quantum  # np.rint rounds halves to even
    r = np.minimum(r, E4M3_MAX)
    return np.where(np.isnan(x), np.nan, np.copysign(r, x))


def attention_forward_fp8(q8, k8, v8, descale_q, descale_k, descale_v, id_q, pos_q, id_kv,
                          pos_kv, causal, scale, row_block=256):
    """O [B,Sq,Hq,d_v] and LSE [B,Hq,Sq] of the FP8 forward.

    The pages define attention in bf16 only; this is an FP8 forward of the
    same computation, the adjacent precision.  Reading taken (the plainest one that
    keeps every product in the 8-bit format):

      inputs      q8, k8, v8 hold E4M3 values; the tensors they stand for are
                  descale_q * q8, descale_k * k8, descale_v * v8
      scores      S_ij = scale * descale_q * descale_k * <q8_i, k8_j>   (exact)
      max, sum    m_i = max_j S_ij over valid j;  p_ij = exp(S_ij - m_i);
                  l_i = sum_j p_ij  (p itself, before any rounding)
      P to E4M3   P8_ij = E4M3(256 p_ij)  (p <= 1, so P8 <= 256 < 448)
      output      O_i = descale_v * sum_j P8_ij v8_j / (256 l_i),
                  LSE_i = m_i + ln l_i;  O_i = 0, LSE_i = -inf without valid j

    The quantisation of P is taken against the row's final maximum (every
    p_ij <= 1), so the result does not depend on how the keys are blocked.
    Everything else is float64."""
    B, Sq, Hq, _ = q8.shape
    _, Skv, Hkv, d_v = v8.shape
    group = Hq // Hkv
    sc = scale * descale_q * descale_k
    o = np.zeros((B, Sq, Hq, d_v))
    lse = np.full((B, Hq, Sq), -np.inf)
    for b in range(B):
        mask = valid_pairs(id_q[b], pos_q[b], id_kv[b], pos_kv[b], causal)
        for h in range(Hq):
            g = h // group
            for r0 in range(0, Sq, row_block):
                r1 = min(Sq, r0 + row_block)
                mrow = mask[r0:r1]
                cols = np.nonzero(mrow.any(axis=0))[0]
                if cols.size == 0:
                    continue
                s = sc * (q8[b, r0:r1, h] @ k8[b, cols, g].T)
                s = np.where(mrow[:, cols], s, -np.inf)
                m = s.max(axis=1)
                fin = np.isfinite(m)
                p = np.zeros_like(s)
                p[fin] = np.exp(s[fin] - m[fin, None])
                l = p.sum(axis=1)
                p8 = e4m3_round(P_SCALE * p)
                out = np.zeros((r1 - r0, d_v))
                out[fin] = descale_v * (p8[fin] @ v8[b, cols, g]) / (P_SCALE * l[fin, None])
                o[b, r0:r1, h] = out
                lse[b, h, r0:r1][fin] = m[fin] + np.log(l[fin])
    return o, lse


def max_logit(q, k, id_q, pos_q, id_kv, pos_kv, causal, scale, bias=None, row_block=256):
    """[B, Hq]: for each batch row and query head the largest S_ij over valid
    (i, j) pairs, in natural units (-inf where no pair is valid).

    TransformerEngine PR #3516 ("[JAX] Align fused attn backward output
    gradient sharding and other test strengthening", Description, item 5.1)
    names max-logit runner cases without defining the output; the reading
    here is the plainest one: the maximum of the same post-scale, post-bias
    logits S_ij that the softmax normalises, taken per (batch row, query
    head) over the pairs the mask keeps."""
    B, Sq, Hq, _ = q.shape
    Hkv = k.shape[2]
    group = Hq // Hkv
    out = np.full((B, Hq), -np.inf)
    for b in range(B):
        mask = valid_pairs(id_q[b], pos_q[b], id_kv[b], pos_kv[b], causal)
        for h in range(Hq):
            g = h // group
            for r0 in range(0, Sq, row_block):
                r1 = min(Sq, r0 + row_block)
                br = None
                if bias is not None:
                    bi, hi = _bias_index(bias.shape, b, h)
                    br = bias[bi, hi, r0:r1]
                cols, _, _, m, _ = _rows_softmax(q[b, r0:r1, h], k[b, :, g], mask[r0:r1],
                                                 scale, br)
                if cols.size:
                    out[b, h] = max(out[b, h], float(m.max()))
    return out


def attention_backward(q, k, v, do, id_q, pos_q, id_kv, pos_kv, causal, scale, bias=None,
                       row_block=256, sink=None):
    """Closed-form gradients (dQ, dK, dV, dBias or None) for the incoming dO.
    With sink logits the probabilities include the sink column (see
    attention_forward); its gradient is sink_gradient().

    The probabilities are recomputed here from Q, K, V (and bias), so the
    backward depends on nothing but the definition.  dBias has the shape of the
    bias and sums dS over every axis the bias broadcasts along."""
    B, Sq, Hq, _ = q.shape
    _, Skv, Hkv, _ = v.shape
    group = Hq // Hkv
    dq = np.zeros(q.shape)
    dk = np.zeros(k.shape)
    dv = np.zeros(v.shape)
    dbias = None if bias is None else np.zeros(bias.shape)
    for b in range(B):
        mask = valid_pairs(id_q[b], pos_q[b], id_kv[b], pos_kv[b], causal)
        for h in range(Hq):
            g = h // group
            for r0 in range(0, Sq, row_block):
                r1 = min(Sq, r0 + row_block)
                br = None
                if bias is not None:
                    bi, hi = _bias_index(bias.shape, b, h)
                    br = bias[bi, hi, r0:r1]
                sk = None if sink is None else float(sink[h])
                cols, _, p, _, _ = _rows_softmax(q[b, r0:r1, h], k[b, :, g], mask[r0:r1],
                                                 scale, br, sk)
                if cols.size == 0:
                    continue
                do_r = do[b, r0:r1, h]
                dp = do_r @ v[b, cols, g].T
                D = (p * dp).sum(axis=1)
                ds = p * (dp - D[:, None])
                dq[b, r0:r1, h] = scale * (ds @ k[b, cols, g])
                dk[b, cols, g] += scale * (ds.T @ q[b, r0:r1, h])
                dv[b, cols, g] += p.T @ do_r
                if dbias is not None:
                    dbias[bi, hi, r0:r1][:, cols] += ds
    return dq, dk, dv, dbias


def sink_gradient(q, k, v, do, id_q, pos_q, id_kv, pos_kv, causal, scale, sink, bias=None,
                  row_block=256):
    """[Hq]: derivative of sum(dO * O) with respect to each head's sink logit.
    The sink column has no value vector, so dP there is 0 and its dS is
    -P_sink,i D_i with D_i = sum_j P_ij dP_ij; summed over batch rows and query
    rows: dsink_h = -sum_{b,i} P_sink,i D_i."""
    B, Sq, Hq, _ = q.shape
    Hkv = v.shape[2]
    group = Hq // Hkv
    out = np.zeros(Hq)
    for b in range(B):
        mask = valid_pairs(id_q[b], pos_q[b], id_kv[b], pos_kv[b], causal)
        for h in range(Hq):
            g = h // group
            for r0 in range(0, Sq, row_block):
                r1 = min(Sq, r0 + row_block)
                br = None
                if bias is not None:
                    bi, hi = _bias_index(bias.shape, b, h)
                    br = bias[bi, hi, r0:r1]
                cols, _, p, m, l = _rows_softmax(q[b, r0:r1, h], k[b, :, g], mask[r0:r1],
                                                 scale, br, float(sink[h]))
                if cols.size == 0:
                    continue
                dp = do[b, r0:r1, h] @ v[b, cols, g].T
                D = (p * dp).sum(axis=1)
                fin = np.isfinite(m)
                p_sink = np.zeros(r1 - r0)
                p_sink[fin] = np.exp(sink[h] - m[fin]) / l[fin]
                out[h] -= float((p_sink * D).sum())
    return out


# --------------------------------------------------------------------------
# Sampled evaluation for full-size checks
# --------------------------------------------------------------------------


def forward_rows(q, k, v, id_q, pos_q, id_kv, pos_kv, causal, scale, b, h, rows, bias=None):
    """O and LSE of the listed query rows of (b, h) only."""
    Hq, Hkv = q.shape[2], v.shape[2]
    g = h // (Hq // Hkv)
    rows = np.asarray(rows)
    mask = valid_pairs(id_q[b][rows], pos_q[b][rows], id_kv[b], pos_kv[b], causal)
    br = None
    if bias is not None:
        bi, hi = _bias_index(bias.shape, b, h)
        br = bias[bi, hi, rows]
    cols, _, p, m, l = _rows_softmax(q[b, rows, h], k[b, :, g], mask, scale, br)
    o = np.zeros((rows.size, v.shape[3]))
    lse = np.full(rows.size, -np.inf)
    if cols.size:
        o = p @ v[b, cols, g]
        fin = np.isfinite(m)
        lse[fin] = m[fin] + np.log(l[fin])
    return o, lse


def backward_dq_rows(q, k, v, do, id_q, pos_q, id_kv, pos_kv, causal, scale, b, h, rows,
                     bias=None):
    """dQ of the listed query rows of (b, h) only (each row needs only its own
    softmax row, so this is exact)."""
    Hq, Hkv = q.shape[2], v.shape[2]
    g = h // (Hq // Hkv)
    rows = np.asarray(rows)
    mask = valid_pairs(id_q[b][rows], pos_q[b][rows], id_kv[b], pos_kv[b], causal)
    br = None
    if bias is not None:
        bi, hi = _bias_index(bias.shape, b, h)
        br = bias[bi, hi, rows]
    cols, _, p, _, _ = _rows_softmax(q[b, rows, h], k[b, :, g], mask, scale, br)
    out = np.zeros((rows.size, q.shape[3]))
    if cols.size:
        dp = do[b, rows, h] @ v[b, cols, g].T
        D = (p * dp).sum(axis=1)
        out = scale * ((p * (dp - D[:, None])) @ k[b, cols, g])
    return out


def backward_dkdv_cols(q, k, v, do, id_q, pos_q, id_kv, pos_kv, causal, scale, b, g, cols,
                       bias=None):
    """dK and dV of the listed key rows of (b, kv-head g).  Every query row that
    attends to one of them is recomputed in full (its softmax needs all of its
    keys), so the result is exact, not an approximation."""
    Hq, Hkv = q.shape[2], v.shape[2]
    group = Hq // Hkv
    cols = np.asarray(cols)
    dk = np.zeros((cols.size, k.shape[3]))
    dv = np.zeros((cols.size, v.shape[3]))
    sel = valid_pairs(id_q[b], pos_q[b], id_kv[b][cols], pos_kv[b][cols], causal)
    rows = np.nonzero(sel.any(axis=1))[0]
    if rows.size == 0:
        return dk, dv
    mask = valid_pairs(id_q[b][rows], pos_q[b][rows], id_kv[b], pos_kv[b], causal)
    for h in range(g * group, (g + 1) * group):
        br = None
        if bias is not None:
            bi, hi = _bias_index(bias.shape, b, h)
            br = bias[bi, hi, rows]
        kc, _, p, _, _ = _rows_softmax(q[b, rows, h], k[b, :, g], mask, scale, br)
        dp = do[b, rows, h] @ v[b, kc, g].T
        D = (p * dp).sum(axis=1)
        ds = p * (dp - D[:, None])
        where = {int(c): n for n, c in enumerate(kc)}
        for t, c in enumerate(cols):
            n = where.get(int(c))
            if n is None:
                continue
            dk[t] += scale * (ds[:, n] @ q[b, rows, h])
            dv[t] += p[:, n] @ do[b, rows, h]
    return dk, dv


# --------------------------------------------------------------------------
# Comparison metric
# --------------------------------------------------------------------------


def rel_frobenius(x, ref):
    """||x - ref||_F / ||ref||_F over the given elements (0 when both vanish)."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref.ravel())
    num = np.linalg.norm((x - ref).ravel())
    if den == 0.0:
        return 0.0 if num == 0.0 else np.inf
    return float(num / den)


def attention_flops(n_valid_pairs_all_heads, d_qk, d_v):
    """Algorithmic FLOPs: forward 2*P*(d_qk + d_v); backward 2*P*(3*d_qk + 2*d_v)
    (the five-GEMM count including the recomputed Q K^T)."""
    P = n_valid_pairs_all_heads
    return 2.0 * P * (d_qk + d_v), 2.0 * P * (3 * d_qk + 2 * d_v)
