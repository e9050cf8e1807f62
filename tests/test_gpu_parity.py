"""GPU parity: the CUDA library (through the C ABI) against the float64 oracle
on the same seeded inputs, element by element (relative Frobenius error over
valid elements, exact zeros / -inf where the definition gives them)."""
import numpy as np
import pytest
import torch

from bwd_tcgen05_tma_gb300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bwd_tcgen05_tma_gb300 import build

    build.build()


def small_cases():
    """Sizes the oracle finishes in seconds that still span several tiles and
    end in a ragged tail."""
    return {
        "tiny": lambda: I.workload("tiny"),
        "bshd_causal_ragged": lambda: I.synth(
            "bshd", B=2, Sq=300, Skv=300, Hq=2, Hkv=2, d_qk=128, d_v=128, layout="HD_HD_HD",
            fmt="BSHD", causal=True, seed=11),
        "bshd_noncausal_cross": lambda: I.synth(
            "bshd_x", B=2, Sq=200, Skv=333, Hq=2, Hkv=1, d_qk=64, d_v=64, layout="HD_HD_HD",
            fmt="BSHD", causal=False, seed=12),
        "thd_gqa_3hd": lambda: I.synth(
            "thd", B=2, Sq=1000, Skv=1000, Hq=4, Hkv=2, d_qk=128, d_v=128, layout="3HD",
            fmt="THD_SEGMENTS", causal=True, seed=13, seg=(40, 400), pad_frac=0.05),
        "cross_bias_192": lambda: I.synth(
            "xb", B=2, Sq=300, Skv=520, Hq=2, Hkv=2, d_qk=192, d_v=128, layout="HD_HD_HD",
            fmt="THD_SEGMENTS", causal=False, seed=14, seg=(60, 200), kv_seg=(60, 300),
            bias_shape=(1, 2, 300, 520)),
        "kvpacked_gqa": lambda: I.synth(
            "kvp", B=1, Sq=700, Skv=700, Hq=4, Hkv=1, d_qk=128, d_v=128, layout="HD_2HD",
            fmt="BSHD", causal=True, seed=15),
        "qk192_v64": lambda: I.synth(
            "q192", B=1, Sq=260, Skv=260, Hq=2, Hkv=2, d_qk=192, d_v=64, layout="HD_HD_HD",
            fmt="THD_SEGMENTS", causal=True, seed=16, seg=(30, 140), pad_frac=0.1),
    }


CASES = small_cases()


def _ref(case):
    from conftest import oracle_full

    return oracle_full(case)


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("force_general", [False, True])
def test_forward_matches_oracle(name, force_general):
    from gpu_util import DevCase, check_forward

    case = CASES[name]()
    ref = _ref(case)
    d = DevCase(case, force_general=force_general)
    o, lse = d.forward()
    check_forward(case, ref, o, lse)
    if force_general:
        assert d.fwd_stats.path == 1


@pytest.mark.parametrize("force_general", [False, True])
def test_forward_many_items_per_cta(force_general):
    """More (query tile, head pair) items than CTAs, so each CTA runs several
    in a row, and key ranges whose last tile is used only in its first half
    (those items take an odd number of 64-key steps)."""
    from gpu_util import DevCase, check_forward

    case = I.synth("thd_many", B=2, Sq=2048, Skv=2048, Hq=32, Hkv=8, d_qk=128, d_v=128,
                   layout="3HD", fmt="THD_SEGMENTS", causal=True, seed=21, seg=(40, 500),
                   pad_frac=0.05)
    ref = _ref(case)
    d = DevCase(case, force_general=force_general)
    o, lse = d.forward()
    check_forward(case, ref, o, lse)


def test_fast_path_taken_for_matching_metadata():
    from gpu_util import DevCase

    d = DevCase(CASES["thd_gqa_3hd"]())
    d.forward()
    assert d.fwd_stats.path == 0 and d.fwd_stats.reason == 1
    d = DevCase(CASES["bshd_causal_ragged"]())
    d.forward()
    assert d.fwd_stats.path == 0 and d.fwd_stats.reason == 0
    d = DevCase(CASES["cross_bias_192"]())
    d.forward()
    assert d.fwd_stats.path == 1 and d.fwd_stats.reason == 3


def test_equal_length_cross_attention_takes_general_path():
    """Sq == Skv but Q and KV segments drawn independently: the general path."""
    from gpu_util import DevCase, check_forward

    case = I.synth("eqx", B=2, Sq=512, Skv=512, Hq=2, Hkv=2, d_qk=128, d_v=128,
                   layout="HD_HD_HD", fmt="THD_SEGMENTS", causal=True, seed=21, seg=(50, 300),
                   kv_seg=(50, 300))
    d = DevCase(case)
    o, lse = d.forward()
    assert d.fwd_stats.path == 1 and d.fwd_stats.reason in (4, 5)
    check_forward(case, _ref(case), o, lse)


def test_derived_positions():
    """Missing segment positions are derived on the device from the ids."""
    from gpu_util import DevCase, check_forward

    case = CASES["thd_gqa_3hd"]()
    d = DevCase(case, with_pos=False)
    o, lse = d.forward()
    assert d.fwd_stats.path == 0
    check_forward(case, _ref(case), o, lse)


def test_cu_seqlens_format():
    from gpu_util import DevCase, check_forward

    base = I.synth("cu", B=1, Sq=900, Skv=900, Hq=2, Hkv=2, d_qk=128, d_v=128,
                   layout="HD_HD_HD", fmt="BSHD", causal=True, seed=22)
    base.fmt = "THD_CU_SEQLENS"
    base.cu_seqlens_q = np.array([0, 130, 130, 500, 777, 860], dtype=np.int32)  # empty segment
    base.cu_seqlens_kv = base.cu_seqlens_q.copy()
    d = DevCase(base)
    o, lse = d.forward()
    assert d.fwd_stats.path == 0
    check_forward(base, _ref(base), o, lse)


# ----------------------------------------------------------------- backward


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("dq_mode", ["deterministic", "atomic"])
def test_backward_matches_oracle(name, dq_mode):
    from gpu_util import DevCase, check_backward

    case = CASES[name]()
    ref = _ref(case)
    d = DevCase(case, dq_mode=dq_mode)
    d.forward()
    g, db = d.backward()
    check_backward(case, ref, g, db)
    expect = 1 if (dq_mode == "deterministic" or case.d_qk > 128) else 0
    assert d.bwd_stats.dq_mode == expect


@pytest.mark.parametrize("shape,window", [("strided", None), ("strided", (90, None)),
                                          ("shifted", None), ("shifted", (90, None))])
def test_general_path_position_shapes(shape, window):
    """Positions that are not offsets from 0 (the general path, reason 6):
    strided (2 x offset, so no chunk has consecutive positions and every chunk
    the band cuts is tested token by token) or shifted by 5 (consecutive, so
    chunk summaries decide the cut chunks), with a causal mask and a causal
    window in position units."""
    from gpu_util import DevCase, check_backward, check_forward

    case = I.synth("pos", B=2, Sq=1000, Skv=1000, Hq=4, Hkv=2, d_qk=128, d_v=128, layout="3HD",
                   fmt="THD_SEGMENTS", causal=True, seed=23, seg=(40, 400), pad_frac=0.05)
    ids = case.q_ids
    starts = np.concatenate([np.ones((ids.shape[0], 1), bool), ids[:, 1:] != ids[:, :-1]], axis=1)
    run = np.cumsum(starts, axis=1)
    offs = np.zeros_like(ids)
    for b in range(ids.shape[0]):
        first = np.maximum.accumulate(np.where(starts[b], np.arange(ids.shape[1]), 0))
        offs[b] = np.arange(ids.shape[1]) - first
    pos = 2 * offs + (run % 3) if shape == "strided" else offs + 5
    pos = np.where(ids != 0, pos, 0).astype(np.int32)
    case.q_pos = pos
    case.kv_pos = pos.copy()
    case.window = window
    ref = _ref(case)
    d = DevCase(case)
    o, lse = d.forward()
    assert d.fwd_stats.path == 1 and d.fwd_stats.reason == 6
    check_forward(case, ref, o, lse)
    g, db = d.backward()
    check_backward(case, ref, g, db)


@pytest.mark.parametrize("name", ["thd_gqa_3hd", "cross_bias_192", "tiny"])
def test_backward_general_path(name):
    from gpu_util import DevCase, check_backward

    case = CASES[name]()
    d = DevCase(case, dq_mode="atomic", force_general=True)
    d.forward()
    g, db = d.backward()
    assert d.bwd_stats.path == 1
    check_backward(case, _ref(case), g, db)


@pytest.mark.parametrize("bias_shape", [(2, 2, 300, 520), (1, 1, 300, 520), (2, 1, 300, 520)])
def test_bias_shapes_and_reduction(bias_shape):
    """dBias per batch/head, and reduced over broadcast batch and head axes."""
    from gpu_util import DevCase, check_backward, check_forward

    case = I.synth("xb", B=2, Sq=300, Skv=520, Hq=4, Hkv=2, d_qk=128, d_v=128,
                   layout="HD_HD_HD", fmt="THD_SEGMENTS", causal=False, seed=31, seg=(60, 200),
                   kv_seg=(60, 300), bias_shape=(bias_shape[0], 4 if bias_shape[1] == 2 else 1,
                                                 300, 520))
    ref = _ref(case)
    d = DevCase(case, dq_mode="deterministic")
    o, lse = d.forward()
    check_forward(case, ref, o, lse)
    g, db = d.backward()
    check_backward(case, ref, g, db)


@pytest.mark.parametrize("dq_mode,bias_shape,d_qk", [
    ("deterministic", (1, 1), 128), ("deterministic", (1, 4), 128), ("deterministic", (2, 1), 128),
    ("atomic", (1, 1), 128), ("deterministic", (1, 1), 192)])
def test_backward_reads_no_stale_workspace(dq_mode, bias_shape, d_qk):
    """The backward reads nothing of its workspace that the same call did not
    write first: filled with 0xFF bytes (NaN as fp32) beforehand, it gives the
    oracle's gradients, including a dBias summed over broadcast batch rows and
    heads through an accumulator that is never cleared."""
    from gpu_util import DevCase, check_backward

    Hq, Hkv = (4, 2) if d_qk == 128 else (2, 2)
    case = I.synth("ws", B=2, Sq=300, Skv=520, Hq=Hq, Hkv=Hkv, d_qk=d_qk, d_v=128,
                   layout="HD_HD_HD", fmt="THD_SEGMENTS", causal=False, seed=33, seg=(60, 200),
                   kv_seg=(60, 300), bias_shape=(bias_shape[0], Hq if bias_shape[1] > 1 else 1,
                                                 300, 520))
    ref = _ref(case)
    d = DevCase(case, dq_mode=dq_mode)
    d.forward()
    d.ws_bwd.fill_(0xFF)
    g, db = d.backward()
    check_backward(case, ref, g, db)


@pytest.mark.parametrize("dq_mode,d_qk", [("deterministic", 192), ("atomic", 128),
                                         ("deterministic", 128)])
def test_bias_rows_not_16_byte_aligned(dq_mode, d_qk):
    """A key count that is not a multiple of 8 leaves bias rows off 16-byte
    boundaries: the bias tile and row loads take their element-wise paths."""
    from gpu_util import DevCase, check_backward, check_forward

    case = I.synth("xu", B=2, Sq=300, Skv=517, Hq=2, Hkv=2, d_qk=d_qk, d_v=128,
                   layout="HD_HD_HD", fmt="THD_SEGMENTS", causal=False, seed=34, seg=(60, 200),
                   kv_seg=(60, 300), bias_shape=(1, 2, 300, 517))
    ref = _ref(case)
    d = DevCase(case, dq_mode=dq_mode)
    o, lse = d.forward()
    check_forward(case, ref, o, lse)
    g, db = d.backward()
    check_backward(case, ref, g, db)


def test_deterministic_mode_bit_reproducible():
    from gpu_util import DevCase

    case = CASES["thd_gqa_3hd"]()
    d = DevCase(case, dq_mode="deterministic")
    d.forward()
    g1, _ = d.backward()
    g1 = {k: v.clone() for k, v in g1.items()}
    g2, _ = d.backward()
    for k in g1:
        assert torch.equal(g1[k].view(torch.int16), g2[k].view(torch.int16)), k


def test_dkdv_dbias_bit_reproducible_in_atomic_mode():
    from gpu_util import DevCase, unpack_grads

    case = I.synth("xb", B=2, Sq=300, Skv=520, Hq=2, Hkv=2, d_qk=128, d_v=128,
                   layout="HD_HD_HD", fmt="THD_SEGMENTS", causal=False, seed=32, seg=(60, 200),
                   kv_seg=(60, 300), bias_shape=(1, 2, 300, 520))
    d = DevCase(case, dq_mode="atomic")
    d.forward()
    g1, db1 = d.backward()
    g1 = {k: v.clone() for k, v in g1.items()}
    db1 = db1.clone()
    g2, db2 = d.backward()
    assert torch.equal(g1["dk"].view(torch.int16), g2["dk"].view(torch.int16))
    assert torch.equal(g1["dv"].view(torch.int16), g2["dv"].view(torch.int16))
    assert torch.equal(db1.view(torch.int16), db2.view(torch.int16))


def test_padding_garbage_isolation():
    """1000.0 in every padded KV position: outputs and real gradients are
    bit-identical to the clean run, and padded tokens get exactly zero grads."""
    from gpu_util import DevCase

    case = I.synth("pad", B=2, Sq=700, Skv=700, Hq=2, Hkv=1, d_qk=128, d_v=128,
                   layout="HD_HD_HD", fmt="THD_SEGMENTS", causal=True, seed=33, seg=(50, 300),
                   pad_frac=0.1)
    clean = DevCase(case)
    o1, l1 = clean.forward()
    o1, l1 = o1.clone(), l1.clone()
    g1, _ = clean.backward()
    g1 = {k: v.clone() for k, v in g1.items()}
    pad = case.kv_ids == 0
    assert pad.sum() > 0
    dirty = I.synth("pad", B=2, Sq=700, Skv=700, Hq=2, Hkv=1, d_qk=128, d_v=128,
                    layout="HD_HD_HD", fmt="THD_SEGMENTS", causal=True, seed=33, seg=(50, 300),
                    pad_frac=0.1)
    dirty.buffers["k"][pad] = 1000.0
    dirty.buffers["v"][pad] = 1000.0
    dd = DevCase(dirty)
    o2, l2 = dd.forward()
    g2, _ = dd.backward()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)
    padt = torch.from_numpy(pad).cuda()
    for k in ("dk", "dv"):
        assert torch.all(g2[k][padt] == 0)
        assert torch.equal(g1[k].view(torch.int16), g2[k].view(torch.int16))
    assert torch.equal(g1["dq"].view(torch.int16), g2["dq"].view(torch.int16))


@pytest.mark.parametrize("name,force_general", [("thd_gqa_3hd", False), ("thd_gqa_3hd", True),
                                                ("bshd_causal_ragged", False)])
def test_backward_reusing_forward_metadata(name, force_general):
    """With metadata_from_forward set, attn_bwd on the forward's workspace skips
    the metadata pass; the gradients are bit-identical to a backward that
    recomputes it, and the reported path is the forward's."""
    from gpu_util import DevCase

    from bwd_tcgen05_tma_gb300 import attn as A

    case = CASES[name]()
    d = DevCase(case, dq_mode="deterministic", force_general=force_general)
    d.forward()
    g_ref, _ = d.backward()
    g_ref = {k: v.clone() for k, v in g_ref.items()}
    path_ref = (d.bwd_stats.path, d.bwd_stats.reason)

    d.params.metadata_from_forward = 1
    ws = d.ws_bwd  # one buffer for both calls
    A.attn_fwd(d.params, d.o, d.lse, ws)
    g, (dq, dk, dv) = d.grad_buffers()
    for _ in range(2):  # the work counters restart on every call
        A.attn_bwd(d.params, d.o, d.do, d.lse, dq, dk, dv, None, ws)
        st, stats = A.attn_read_status(ws)
        assert st == 0
        assert (stats.path, stats.reason) == path_ref
        for k in g_ref:
            assert torch.equal(g[k].view(torch.int16), g_ref[k].view(torch.int16)), k


@pytest.mark.parametrize("force_general", [False, True])
def test_many_rows_match_single_row_calls(force_general):
    """160 rows of 2100 tokens: more 1024-token metadata blocks than the
    metadata kernel's grid holds, so every pass strides over its units, and
    segment bounds carry across blocks.  Rows are independent: each row's
    outputs and gradients equal, bit for bit, those of a call on that row
    alone (whose parity with the oracle the other tests cover)."""
    import copy

    from gpu_util import DevCase

    big = I.synth("rows", B=160, Sq=2100, Skv=2100, Hq=1, Hkv=1, d_qk=64, d_v=64,
                  layout="HD_HD_HD", fmt="THD_SEGMENTS", causal=True, seed=51, seg=(64, 2048),
                  pad_frac=0.05)
    d = DevCase(big, force_general=force_general)
    o, lse = d.forward()
    g, _ = d.backward()
    assert d.fwd_stats.path == (1 if force_general else 0)
    for b in (0, 77, 159):
        one = copy.copy(big)
        one.B = 1
        one.buffers = {k: v[b:b + 1] for k, v in big.buffers.items()}
        one.do = big.do[b:b + 1]
        for f in ("q_ids", "q_pos", "kv_ids", "kv_pos"):
            setattr(one, f, getattr(big, f)[b:b + 1])
        s = DevCase(one, force_general=force_general)
        o1, l1 = s.forward()
        g1, _ = s.backward()
        assert torch.equal(o.view(160, 2100, -1)[b].view(torch.int16),
                           o1.view(2100, -1).view(torch.int16)), b
        assert torch.equal(lse[b], l1[0]), b
        for k in g1:
            assert torch.equal(g[k][b].view(torch.int16), g1[k][0].view(torch.int16)), (k, b)


@pytest.mark.parametrize("name", ["tiny", "thd_gqa_3hd", "cross_bias_192", "bshd_causal_ragged",
                                  "qk192_v64"])
def test_max_logit_matches_oracle(name):
    """The optional max-logit output of the forward against the oracle's; the
    forward's other outputs are unchanged by requesting it."""
    from conftest import oracle_metadata, oracle_qkv
    from gpu_util import DevCase
    from oracle import attn_ref as R

    case = CASES[name]()
    d = DevCase(case)
    o0, l0 = d.forward()
    o0, l0 = o0.clone(), l0.clone()
    ml = torch.full((case.B, case.Hq), 123.0, dtype=torch.float32, device="cuda")
    d.params.max_logit = ml.data_ptr()
    o1, l1 = d.forward()
    assert torch.equal(o0.view(torch.int16), o1.view(torch.int16))
    assert torch.equal(l0, l1)
    q, k, _ = oracle_qkv(case)
    qi, qp, ki, kp = oracle_metadata(case)
    bias = None if case.bias is None else case.bias.astype(np.float64)
    ref = R.max_logit(q, k, qi, qp, ki, kp, case.causal, case.scale, bias)
    got = ml.cpu().numpy().astype(np.float64)
    assert np.array_equal(np.isfinite(got), np.isfinite(ref))
    fin = np.isfinite(ref)
    np.testing.assert_allclose(got[fin], ref[fin], rtol=1e-4, atol=1e-4)
    assert np.all(got[~fin] == -np.inf)


@pytest.mark.parametrize("name", ["tiny", "thd_gqa_3hd", "cross_bias_192"])
def test_sink_attention_matches_oracle(name):
    """Per-head sink logits: O, LSE (a row without valid keys gets its head's
    sink), dQ/dK/dV/dBias, and the sink gradient against the oracle; the sink
    gradient reproduces itself bit for bit."""
    from conftest import oracle_metadata, oracle_qkv
    from gpu_util import DevCase, check_backward, check_forward
    from oracle import attn_ref as R

    case = CASES[name]()
    rng = np.random.default_rng(21)
    sink_h = (rng.standard_normal(case.Hq) * 1.5 + 0.5).astype(np.float32)
    sink = torch.from_numpy(sink_h).cuda()
    dsink = torch.full((case.Hq,), float("nan"), dtype=torch.float32, device="cuda")
    d = DevCase(case)
    d.params.sink = sink.data_ptr()
    d.params.dsink = dsink.data_ptr()
    d.ws_bwd = torch.zeros(max(_bwd_ws_size(d.params), 256), dtype=torch.uint8, device="cuda")

    q, k, v = oracle_qkv(case)
    qi, qp, ki, kp = oracle_metadata(case)
    bias = None if case.bias is None else case.bias.astype(np.float64)
    do = case.do.astype(np.float64)
    s64 = sink_h.astype(np.float64)
    o_r, lse_r = R.attention_forward(q, k, v, qi, qp, ki, kp, case.causal, case.scale, bias,
                                     sink=s64)
    dq_r, dk_r, dv_r, db_r = R.attention_backward(q, k, v, do, qi, qp, ki, kp, case.causal,
                                                  case.scale, bias, sink=s64)
    ds_r = R.sink_gradient(q, k, v, do, qi, qp, ki, kp, case.causal, case.scale, s64, bias)
    ref = {"o": o_r, "lse": lse_r, "dq": dq_r, "dk": dk_r, "dv": dv_r, "dbias": db_r}

    o, lse = d.forward()
    check_forward(case, ref, o, lse)
    g, db = d.backward()
    check_backward(case, ref, g, db)
    got = dsink.cpu().numpy().astype(np.float64)
    # the sum of per-row terms may cancel: bound the error by their magnitudes
    D = (do * o_r).sum(axis=3)  # [B, Sq, Hq]
    mag = np.abs(np.exp(s64[None, :, None] - lse_r) * D.transpose(0, 2, 1)).sum(axis=(0, 2))
    assert np.all(np.abs(got - ds_r) <= 1e-2 * mag + 1e-6), (got, ds_r, mag)
    first = dsink.clone()
    d.backward()
    assert torch.equal(first, dsink)


def _bwd_ws_size(params):
    from bwd_tcgen05_tma_gb300 import attn as A

    return A.attn_bwd_workspace_size(params)


def test_backward_gradients_only_16_byte_aligned():
    """Gradient buffers that start 16 bytes past a 32-byte boundary (the ABI
    asks for 16): the epilogues then take their 16-byte stores, and the
    gradients are the bits of the aligned call."""
    from gpu_util import DevCase

    from bwd_tcgen05_tma_gb300 import attn as A

    case = CASES["thd_gqa_3hd"]()
    d = DevCase(case, dq_mode="deterministic")
    d.forward()
    g_ref, _ = d.backward()
    ref = g_ref["dqkv"].clone()
    W = ref.shape[1]
    big = torch.full((ref.numel() + 16,), float("nan"), dtype=torch.bfloat16, device="cuda")
    assert big.data_ptr() % 32 == 0
    dqkv = big[8:8 + ref.numel()].view(ref.shape)  # 16 bytes past the boundary
    assert dqkv.data_ptr() % 32 == 16
    A.attn_bwd(d.params, d.o, d.do, d.lse, dqkv, None, None, None, d.ws_bwd)
    st, _ = A.attn_read_status(d.ws_bwd)
    assert st == 0 and W == dqkv.shape[1]
    assert torch.equal(dqkv.view(torch.int16), ref.view(torch.int16))
