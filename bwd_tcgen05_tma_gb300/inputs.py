"""Seeded synthetic inputs for the attention workloads.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic.  Both the CUDA path and the float64 oracle consume what
it returns: tensors are drawn in float32 from ``numpy.random.default_rng(seed)``
and rounded to bfloat16 (or, for cases of the fp16 element type, to float16;
round to nearest even), so both sides see exactly the same 16-bit values.

Workloads (one seed each, sizes as named):

* ``tiny``      B=2, S=128, Hq=Hkv=2, D=64, separate Q/K/V; every row packs two
                segments of random length (ids 1, 2, positions restarting at 0)
                and a padding tail (id 0) of U[1,16] tokens; causal inside
                segments.
* ``bshd``      B=4, S=2048, Hq=Hkv=16, D=128, separate Q/K/V, dense causal.
* ``thd_gqa``   2 rows x 8192 tokens; a 5 % padding tail (410 tokens, id 0);
                the rest filled with segments of length U[64,2048] (the last
                one truncated); Hq=32, Hkv=8, D=128; packed QKV; causal.
* ``cross_bias`` B=2, Sq=4096, Skv=8192, Hq=Hkv=16, d_qk=192, d_v=128; Q and KV
                segments drawn independently with lengths U[128,4096] (last one
                truncated, ids 1..n in order, no padding); not causal; bias
                [1,16,4096,8192] ~ N(0, 0.5^2) with its gradient.
* ``long_kv``   B=1, S=32768, Hq=64, Hkv=8, D=128, packed KV, dense causal.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

# ----------------------------------------------------------------- bf16 bits


def bf16_bits(x):
    """float32 array -> uint16 bf16 bit patterns, round to nearest even
    (NaN -> the canonical quiet NaN)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    r = u + np.uint32(0x7FFF)
    r += (u >> np.uint32(16)) & np.uint32(1)
    r >>= np.uint32(16)
    out = r.astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = 0x7FC0
    return out


def bf16_to_f32(bits):
    """uint16 bf16 bit patterns -> float32 values."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def bf16_round(x):
    """float32 values rounded to the nearest bf16 value (kept as float32)."""
    return bf16_to_f32(bf16_bits(x))


def f16_round(x):
    """float32 values rounded to the nearest fp16 value (kept as float32;
    NumPy's float16 conversion rounds to nearest even)."""
    return np.asarray(x, dtype=np.float32).astype(np.float16).astype(np.float32)


def e4m3_codes(x):
    """E4M3 codes (uint8) of float32 values within +-448, by PyTorch's
    float8_e4m3fn conversion (round to nearest even)."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def e4m3_value(codes):
    """float32 values of E4M3 codes."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.float().numpy()


def round_to(x, dtype):
    """Nearest value of the element type ("bf16", "fp16" or "fp8_e4m3"), as float32."""
    if dtype == "fp8_e4m3":
        return e4m3_value(e4m3_codes(x))
    return bf16_round(x) if dtype == "bf16" else f16_round(x)


# ----------------------------------------------------------------- metadata


def fill_segments(rng, n_tokens, lo, hi):
    """Segment lengths drawn U[lo, hi] until n_tokens are covered; the last
    segment is truncated to fit."""
    lens = []
    left = n_tokens
    while left > 0:
        L = int(rng.integers(lo, hi + 1))
        L = min(L, left)
        lens.append(L)
        left -= L
    return lens


def ids_pos_from_lengths(lens, total):
    """Segment k (0-based) gets id k+1 and positions 0..len-1; the remainder up
    to `total` is padding (id 0, position counting from 0)."""
    ids = np.zeros(total, dtype=np.int32)
    pos = np.zeros(total, dtype=np.int32)
    t = 0
    for k, L in enumerate(lens):
        ids[t : t + L] = k + 1
        pos[t : t + L] = np.arange(L, dtype=np.int32)
        t += L
    if t < total:
        pos[t:] = np.arange(total - t, dtype=np.int32)
    return ids, pos


# ----------------------------------------------------------------- case


@dataclass
class Case:
    name: str
    B: int
    Sq: int
    Skv: int
    Hq: int
    Hkv: int
    d_qk: int
    d_v: int
    layout: str  # "3HD" | "HD_2HD" | "HD_HD_HD"
    fmt: str  # "BSHD" | "THD_SEGMENTS" | "THD_CU_SEQLENS"
    causal: bool
    scale: float
    seed: int
    buffers: dict = field(default_factory=dict)  # float32 arrays holding bf16 values
    do: np.ndarray | None = None  # [B, Sq, Hq, d_v]
    q_ids: np.ndarray | None = None  # [B, Sq] int32
    q_pos: np.ndarray | None = None
    kv_ids: np.ndarray | None = None
    kv_pos: np.ndarray | None = None
    cu_seqlens_q: np.ndarray | None = None
    cu_seqlens_kv: np.ndarray | None = None
    bias: np.ndarray | None = None  # [bias_b, bias_h, Sq, Skv]
    window: tuple | None = None  # band (left, right) in positions, None for an open side
    bottom_right: bool = False  # positions aligned by Skv - Sq
    dtype: str = "bf16"  # element type of the 16-bit tensors: "bf16" or "fp16"

    @property
    def mask(self):
        has_pad = self.fmt != "BSHD" or self.q_ids is not None
        if has_pad:
            return "PADDING_CAUSAL" if self.causal else "PADDING"
        return "CAUSAL" if self.causal else "NONE"


def _normal_bf16(rng, shape, std=1.0, dtype="bf16"):
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return round_to(x, dtype)


def make_buffers(rng, layout, B, Sq, Skv, Hq, Hkv, d_qk, d_v, dtype="bf16"):
    """Raw token-major input buffers of the layout, N(0,1) rounded to the
    element type (bf16 unless dtype is "fp16")."""
    def nrm(shape):
        return _normal_bf16(rng, shape, dtype=dtype)

    if layout == "3HD":
        assert Sq == Skv
        return {"qkv": nrm((B * Sq, Hq * d_qk + Hkv * d_qk + Hkv * d_v))}
    if layout == "HD_2HD":
        assert d_qk == d_v
        return {
            "q": nrm((B * Sq, Hq * d_qk)),
            "kv": nrm((B * Skv, 2, Hkv, d_v)),
        }
    return {
        "q": nrm((B, Sq, Hq, d_qk)),
        "k": nrm((B, Skv, Hkv, d_qk)),
        "v": nrm((B, Skv, Hkv, d_v)),
    }


def synth(name, *, B, Sq, Skv, Hq, Hkv, d_qk, d_v, layout, fmt, causal, seed,
          seg=None, kv_seg=None, pad_frac=0.0, pad_range=None, two_segments=False,
          bias_shape=None, bias_std=0.5, scale=None, dtype="bf16"):
    """General seeded case builder.

    seg / kv_seg: (lo, hi) segment length ranges for Q / KV (kv_seg None means
    the KV metadata equals the Q metadata).  pad_frac: fraction of each row
    left as a padding tail.  two_segments: the tiny-case recipe (padding tail
    U[pad_range], then two segments of random length)."""
    rng = np.random.default_rng(seed)
    c = Case(name=name, B=B, Sq=Sq, Skv=Skv, Hq=Hq, Hkv=Hkv, d_qk=d_qk, d_v=d_v,
             layout=layout, fmt=fmt, causal=causal, seed=seed,
             scale=(1.0 / math.sqrt(d_qk)) if scale is None else scale, dtype=dtype)
    if fmt == "THD_SEGMENTS":
        qi = np.zeros((B, Sq), np.int32)
        qp = np.zeros((B, Sq), np.int32)
        ki = np.zeros((B, Skv), np.int32)
        kp = np.zeros((B, Skv), np.int32)
        for b in range(B):
            if two_segments:
                lo, hi = pad_range
                pad = int(rng.integers(lo, hi + 1))
                L1 = int(rng.integers(1, Sq - pad))  # U[1, Sq-1-pad]
                lens = [L1, Sq - pad - L1]
            else:
                pad = int(round(pad_frac * Sq))
                lens = fill_segments(rng, Sq - pad, *seg)
            qi[b], qp[b] = ids_pos_from_lengths(lens, Sq)
            if kv_seg is None:
                ki[b], kp[b] = qi[b], qp[b]
            else:
                kpad = int(round(pad_frac * Skv))
                klens = fill_segments(rng, Skv - kpad, *kv_seg)
                ki[b], kp[b] = ids_pos_from_lengths(klens, Skv)
        c.q_ids, c.q_pos, c.kv_ids, c.kv_pos = qi, qp, ki, kp
    c.buffers = make_buffers(rng, layout, B, Sq, Skv, Hq, Hkv, d_qk, d_v, dtype)
    # dO and the bias stay 16-bit when Q / K / V are E4M3 (the FP8 path is a
    # forward; O is bf16)
    dt16 = "bf16" if dtype == "fp8_e4m3" else dtype
    c.do = _normal_bf16(rng, (B, Sq, Hq, d_v), dtype=dt16)
    if bias_shape is not None:
        c.bias = _normal_bf16(rng, bias_shape, std=bias_std, dtype=dt16)
    return c


def workload(name, seed=None):
    """The five named workloads at their full sizes."""
    if name == "tiny":
        return synth("tiny", B=2, Sq=128, Skv=128, Hq=2, Hkv=2, d_qk=64, d_v=64,
                     layout="HD_HD_HD", fmt="THD_SEGMENTS", causal=True,
                     seed=0 if seed is None else seed, two_segments=True, pad_range=(1, 16))
    if name == "bshd":
        return synth("bshd", B=4, Sq=2048, Skv=2048, Hq=16, Hkv=16, d_qk=128, d_v=128,
                     layout="HD_HD_HD", fmt="BSHD", causal=True,
                     seed=2 if seed is None else seed)
    if name == "thd_gqa":
        return synth("thd_gqa", B=2, Sq=8192, Skv=8192, Hq=32, Hkv=8, d_qk=128, d_v=128,
                     layout="3HD", fmt="THD_SEGMENTS", causal=True,
                     seed=3 if seed is None else seed, seg=(64, 2048), pad_frac=410 / 8192)
    if name == "cross_bias":
        return synth("cross_bias", B=2, Sq=4096, Skv=8192, Hq=16, Hkv=16, d_qk=192, d_v=128,
                     layout="HD_HD_HD", fmt="THD_SEGMENTS", causal=False,
                     seed=4 if seed is None else seed, seg=(128, 4096), kv_seg=(128, 4096),
                     bias_shape=(1, 16, 4096, 8192), bias_std=0.5)
    if name == "long_kv":
        return synth("long_kv", B=1, Sq=32768, Skv=32768, Hq=64, Hkv=8, d_qk=128, d_v=128,
                     layout="HD_2HD", fmt="BSHD", causal=True,
                     seed=5 if seed is None else seed)
    raise KeyError(name)


WORKLOADS = ("tiny", "bshd", "thd_gqa", "cross_bias", "long_kv")
