"""The seeded input generator: bf16 rounding and the workload recipes."""
import numpy as np
import torch

from bwd_tcgen05_tma_gb300 import inputs as I


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(100000) * 10.0 ** rng.integers(-8, 8, 100000)).astype(np.float32)
    x[:4] = [0.0, -0.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8]  # ties round to even
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(I.bf16_bits(x), ref)
    np.testing.assert_array_equal(I.bf16_round(x),
                                  torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_tiny_recipe():
    c = I.workload("tiny")
    assert c.q_ids.shape == (2, 128) and c.layout == "HD_HD_HD" and c.causal
    for b in range(2):
        ids = c.q_ids[b]
        pad = int((ids == 0).sum())
        assert 1 <= pad <= 16 and np.all(ids[128 - pad:] == 0)
        assert set(np.unique(ids[:128 - pad])) == {1, 2}
        assert np.all(np.diff(ids[:128 - pad]) >= 0)
        for s in (1, 2):
            np.testing.assert_array_equal(c.q_pos[b][ids == s], np.arange((ids == s).sum()))
    assert np.array_equal(c.q_ids, c.kv_ids) and np.array_equal(c.q_pos, c.kv_pos)


def test_thd_recipe_small_seed_stable():
    c = I.synth("t", B=2, Sq=8192, Skv=8192, Hq=2, Hkv=1, d_qk=8, d_v=8, layout="3HD",
                fmt="THD_SEGMENTS", causal=True, seed=3, seg=(64, 2048), pad_frac=410 / 8192)
    for b in range(2):
        ids = c.q_ids[b]
        assert int((ids == 0).sum()) == 410 and np.all(ids[-410:] == 0)
        lens = np.bincount(ids[ids > 0])[1:]
        assert np.all(lens[:-1] >= 64) and np.all(lens <= 2048)
    assert c.buffers["qkv"].shape == (2 * 8192, 2 * 8 + 8 + 8)
    c2 = I.synth("t", B=2, Sq=8192, Skv=8192, Hq=2, Hkv=1, d_qk=8, d_v=8, layout="3HD",
                 fmt="THD_SEGMENTS", causal=True, seed=3, seg=(64, 2048), pad_frac=410 / 8192)
    assert np.array_equal(c.buffers["qkv"], c2.buffers["qkv"])


def test_cross_recipe_independent_metadata():
    c = I.synth("x", B=2, Sq=4096, Skv=8192, Hq=1, Hkv=1, d_qk=8, d_v=8, layout="HD_HD_HD",
                fmt="THD_SEGMENTS", causal=False, seed=4, seg=(128, 4096), kv_seg=(128, 4096),
                bias_shape=(1, 1, 4096, 8192))
    assert c.q_ids.shape == (2, 4096) and c.kv_ids.shape == (2, 8192)
    assert np.all(c.q_ids > 0) and np.all(c.kv_ids > 0)
    assert abs(float(c.bias.std()) - 0.5) < 0.01


def test_fp16_inputs_are_fp16_values():
    """Cases of the fp16 element type hold float32 copies of fp16 values
    (exactly representable, so both sides read the same numbers)."""
    c = I.synth("f", B=1, Sq=64, Skv=64, Hq=2, Hkv=1, d_qk=64, d_v=64, layout="HD_HD_HD",
                fmt="BSHD", causal=True, seed=3, dtype="fp16", bias_shape=(1, 2, 64, 64))
    for x in (c.buffers["q"], c.buffers["k"], c.buffers["v"], c.do, c.bias):
        assert np.array_equal(x.astype(np.float16).astype(np.float32), x)
    assert c.dtype == "fp16"
    assert np.array_equal(I.f16_round(np.float32([1.0 + 2.0 ** -11, 65504.0])),
                          np.float32([1.0, 65504.0]))
