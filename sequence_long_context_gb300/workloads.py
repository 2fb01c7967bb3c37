"""Seeded synthetic workloads for sequence-parallel attention.

This module only draws inputs: shapes, seeded N(0,1) tensors and packed-segment
boundaries. It holds none of the attention arithmetic, so the CUDA path, the
CPU oracle, the tests and the benchmark can all take their inputs from here
without sharing any of the method's computation.

Workload shapes follow the problem statements on the pages this library
implements:
  * the ring sliding-window example shape B=2, S=8192, H=32, D=128 with
    window 1000 ("ring-sliding-window-attention" README, non-varlen example);
  * the USP hybrid example with ulysses degree 2 x ring degree 4 (YunChang
    README, "2. Usage");
  * zigzag and stripe layouts (YunChang README "2. Usage"; "Long Context
    Attention" notes, "Solution" and "Zig-Zag Attention");
  * packed variable-length batches described by a global cu_seqlens
    ("ring-sliding-window-attention" README, varlen example).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import torch

LAYOUTS = ("contiguous", "zigzag", "stripe")


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int            # batch (dense) or number of segments (packed; derived)
    S: int            # sequence length (dense) or total packed tokens T
    Hq: int
    Hkv: int
    D: int
    dtype: str        # "bf16" | "fp32"
    causal: bool
    window: int       # <= 0: no window; else number of visible keys incl. itself
    sink_tokens: int
    cp: int           # ring degree (virtual ranks)
    ud: int           # ulysses degree
    layout: str       # contiguous | zigzag | stripe
    varlen: bool = False
    seg_lo: int = 0   # packed segment length range (inclusive), varlen only
    seg_hi: int = 0
    input_scale: float = 1.0
    backward: bool = True

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five problem shapes plus the causal zigzag sweep used for the metric.
WORKLOADS: Dict[str, Workload] = {
    "tiny_zigzag_cp4": Workload(
        "tiny_zigzag_cp4", B=1, S=256, Hq=2, Hkv=2, D=64, dtype="fp32",
        causal=True, window=0, sink_tokens=0, cp=4, ud=1, layout="zigzag"),
    "usp_ud2_ring4_s8k": Workload(
        "usp_ud2_ring4_s8k", B=2, S=8192, Hq=32, Hkv=32, D=128, dtype="bf16",
        causal=True, window=0, sink_tokens=0, cp=4, ud=2, layout="zigzag"),
    "gqa_stripe_cp8_s32k": Workload(
        "gqa_stripe_cp8_s32k", B=1, S=32768, Hq=32, Hkv=8, D=128, dtype="bf16",
        causal=True, window=0, sink_tokens=0, cp=8, ud=1, layout="stripe",
        input_scale=1.0 / math.sqrt(2.0)),
    "swa_w1000_cp8_s8k": Workload(
        "swa_w1000_cp8_s8k", B=2, S=8192, Hq=32, Hkv=32, D=128, dtype="bf16",
        causal=True, window=1000, sink_tokens=0, cp=8, ud=1,
        layout="contiguous", backward=False),
    "swa_w1000_sink4_cp8_s8k": Workload(
        "swa_w1000_sink4_cp8_s8k", B=2, S=8192, Hq=32, Hkv=32, D=128,
        dtype="bf16", causal=True, window=1000, sink_tokens=4, cp=8, ud=1,
        layout="contiguous", backward=False),
    # the same sliding-window + sink problem as a training step (forward and
    # backward), the ring sliding-window README's use case (LM training)
    "swa_w1000_sink4_cp8_s8k_train": Workload(
        "swa_w1000_sink4_cp8_s8k_train", B=2, S=8192, Hq=32, Hkv=32, D=128,
        dtype="bf16", causal=True, window=1000, sink_tokens=4, cp=8, ud=1,
        layout="contiguous", backward=True),
    "varlen_zigzag_cp8_t128k": Workload(
        "varlen_zigzag_cp8_t128k", B=0, S=131072, Hq=32, Hkv=8, D=128,
        dtype="bf16", causal=True, window=0, sink_tokens=0, cp=8, ud=1,
        layout="zigzag", varlen=True, seg_lo=256, seg_hi=16384),
}
for _s in (8192, 16384, 32768, 65536, 131072):
    _n = f"sweep_zigzag_cp8_s{_s // 1024}k"
    WORKLOADS[_n] = Workload(
        _n, B=1, S=_s, Hq=32, Hkv=8, D=128, dtype="bf16", causal=True,
        window=0, sink_tokens=0, cp=8, ud=1, layout="zigzag")


def draw_cu_seqlens(T: int, lo: int, hi: int, seed: int) -> torch.Tensor:
    """Segment boundaries of a packed batch of T tokens.

    Lengths are drawn uniform in [lo, hi] (inclusive) until they cover T; the
    last segment is cut so the lengths sum to exactly T. Returns int32
    [nseq + 1] starting at 0 and ending at T.
    """
    g = torch.Generator().manual_seed(seed + 7919)
    bounds = [0]
    while bounds[-1] < T:
        L = int(torch.randint(lo, hi + 1, (1,), generator=g).item())
        bounds.append(min(T, bounds[-1] + L))
    return torch.tensor(bounds, dtype=torch.int32)


def torch_dtype(name: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "fp32": torch.float32}[name]


def make_inputs(w: Workload, seed: int = 0, device: str = "cpu",
                with_grad: Optional[bool] = None) -> Dict[str, torch.Tensor]:
    """Seeded q, k, v (and dout) in natural token order.

    Dense shapes are [B, S, H, D]; packed shapes are [T, H, D] plus
    cu_seqlens. Values are N(0,1) drawn in fp32 (times the workload's input
    scale) and then rounded to the workload dtype, so every consumer sees the
    same rounded values.
    """
    if with_grad is None:
        with_grad = w.backward
    g = torch.Generator(device=device).manual_seed(seed)
    dt = torch_dtype(w.dtype)
    if w.varlen:
        qs, ks = (w.S, w.Hq, w.D), (w.S, w.Hkv, w.D)
    else:
        qs, ks = (w.B, w.S, w.Hq, w.D), (w.B, w.S, w.Hkv, w.D)

    def rnd(shape, scale=1.0):
        x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        if scale != 1.0:
            x.mul_(scale)
        return x.to(dt)

    out = {
        "q": rnd(qs, w.input_scale),
        "k": rnd(ks, w.input_scale),
        "v": rnd(ks, w.input_scale),
    }
    if with_grad:
        out["dout"] = rnd(qs)
    if w.varlen:
        out["cu_seqlens"] = draw_cu_seqlens(w.S, w.seg_lo, w.seg_hi, seed)
    return out


def n_segments(w: Workload, inputs: Dict[str, torch.Tensor]) -> int:
    if w.varlen:
        return int(inputs["cu_seqlens"].numel() - 1)
    return w.B


@dataclasses.dataclass(frozen=True)
class DecodeWorkload:
    """One decoding step: the newest Tq tokens against a KV cache of S keys
    sharded over cp ranks (rank-major contiguous), each shard cut into
    `splits` pieces whose partials are merged in tree order."""
    name: str
    B: int
    Tq: int
    S: int
    Hq: int
    Hkv: int
    D: int
    cp: int
    splits: int
    causal: bool = True

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def kv_bytes(self) -> int:
        return 2 * self.B * self.S * self.Hkv * self.D * 2


# The pages give no decode shape; this one reuses the GQA sweep's heads
# (32 query / 8 KV heads, D = 128) and its longest sequence as the cache,
# sharded over the same 8-way ring, one new token for 8 sequences.
DECODE_WORKLOADS: Dict[str, DecodeWorkload] = {
    "decode_gqa_b8_s128k_cp8": DecodeWorkload(
        "decode_gqa_b8_s128k_cp8", B=8, Tq=1, S=131072, Hq=32, Hkv=8, D=128,
        cp=8, splits=4),
}


def make_decode_inputs(w: DecodeWorkload, seed: int = 0, device: str = "cpu"
                       ) -> Dict[str, torch.Tensor]:
    """Seeded bf16 q [B,Tq,Hq,D] and cache k, v [B,S,Hkv,D] (N(0,1) drawn in
    fp32, then rounded)."""
    g = torch.Generator(device=device).manual_seed(seed)

    def rnd(shape):
        return torch.randn(shape, generator=g, device=device,
                           dtype=torch.float32).to(torch.bfloat16)

    return {"q": rnd((w.B, w.Tq, w.Hq, w.D)),
            "k": rnd((w.B, w.S, w.Hkv, w.D)),
            "v": rnd((w.B, w.S, w.Hkv, w.D))}
