"""Seeded synthetic inputs shared by the CUDA path, its tests and the oracle.

This module holds no attention arithmetic: it only draws random numbers and
casts them to the storage type, so that the CUDA kernels and the CPU oracle can
be fed the very same tensors.

Recipe (one ``torch.Generator`` per call, seeded; draws happen in a fixed order):

* prefill: ``q [B,T,Hq,D]``, ``k [B,T,Hkv,D]``, ``v [B,T,Hkv,D]`` ~ N(0,1) drawn in
  fp32 in the order q, k, v, then ``sink [Hq]`` fp32 (N(0,1), or U(-4,4)).
  Optionally every ``peaky_every``-th key row (1-based: rows j with
  ``(j+1) % peaky_every == 0``) is multiplied by ``peaky_scale`` in fp32 before
  the cast, which makes a few scores much larger than the rest.  q, k, v are
  then rounded to the storage dtype (round-to-nearest-even for bf16).
* decode: ``q [B,Hq,D]``, ``k_ring [B,Hkv,W,D]``, ``v_ring [B,Hkv,W,D]``,
  ``sink [Hq]`` in that order, then ``pos [B]`` int64 uniform in
  ``[pos_lo, pos_hi)``.
* verify (L drafted tokens): ``q [B,L,Hq,D]``, ``k_new [B,L,Hkv,D]``,
  ``v_new [B,L,Hkv,D]``, ``k_ring``, ``v_ring [B,Hkv,W,D]``, ``sink [Hq]``, then
  ``pos [B]`` int64 uniform in ``[pos_lo, pos_hi)``.

The model these shapes come from (MiMo-V2-Flash technical report summary,
"core method": 128-token sliding window, GQA, learnable per-head sink) fixes no
value distribution; N(0,1) is the plain choice.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass
class PrefillInputs:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    sink: torch.Tensor


@dataclass
class DecodeInputs:
    q: torch.Tensor
    k_ring: torch.Tensor
    v_ring: torch.Tensor
    sink: torch.Tensor
    pos: torch.Tensor


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def prefill_inputs(B: int, T: int, Hq: int, Hkv: int, D: int, *, seed: int = 0,
                   dtype: torch.dtype = torch.bfloat16, device="cpu",
                   sink_dist: str = "normal", peaky_every: int = 0,
                   peaky_scale: float = 8.0) -> PrefillInputs:
    """Draw one layer's prefill inputs (see module docstring for the recipe)."""
    g = _gen(seed, device)
    f32 = torch.float32
    q = torch.randn(B, T, Hq, D, generator=g, device=device, dtype=f32)
    k = torch.randn(B, T, Hkv, D, generator=g, device=device, dtype=f32)
    v = torch.randn(B, T, Hkv, D, generator=g, device=device, dtype=f32)
    if sink_dist == "normal":
        sink = torch.randn(Hq, generator=g, device=device, dtype=f32)
    elif sink_dist == "uniform4":
        sink = torch.rand(Hq, generator=g, device=device, dtype=f32) * 8.0 - 4.0
    else:
        raise ValueError(f"unknown sink_dist {sink_dist!r}")
    if peaky_every:
        k[:, peaky_every - 1::peaky_every] *= peaky_scale
    return PrefillInputs(q.to(dtype), k.to(dtype), v.to(dtype), sink)


def hybrid_block_inputs(T: int, Hq: int, Hkv: int, D: int, *, n_swa: int = 5,
                        n_ga: int = 1, seed: int = 0, dtype=torch.bfloat16,
                        device="cpu") -> list[PrefillInputs]:
    """Independent inputs for each layer of one hybrid block, layer order
    (n_swa sliding-window layers, then n_ga global layers); layer l uses seed+l."""
    return [prefill_inputs(1, T, Hq, Hkv, D, seed=seed + l, dtype=dtype, device=device)
            for l in range(n_swa + n_ga)]


def decode_inputs(B: int, Hq: int, Hkv: int, D: int, W: int, *, seed: int = 0,
                  dtype: torch.dtype = torch.bfloat16, device="cpu",
                  pos_lo: int = 128, pos_hi: int = 262144) -> DecodeInputs:
    """Draw decode inputs: one query token per sequence and a full W-slot ring."""
    g = _gen(seed, device)
    f32 = torch.float32
    q = torch.randn(B, Hq, D, generator=g, device=device, dtype=f32)
    k_ring = torch.randn(B, Hkv, W, D, generator=g, device=device, dtype=f32)
    v_ring = torch.randn(B, Hkv, W, D, generator=g, device=device, dtype=f32)
    sink = torch.randn(Hq, generator=g, device=device, dtype=f32)
    pos = torch.randint(pos_lo, pos_hi, (B,), generator=g, device=device, dtype=torch.int64)
    return DecodeInputs(q.to(dtype), k_ring.to(dtype), v_ring.to(dtype), sink, pos)


@dataclass
class VerifyInputs:
    q: torch.Tensor
    k_new: torch.Tensor
    v_new: torch.Tensor
    k_ring: torch.Tensor
    v_ring: torch.Tensor
    sink: torch.Tensor
    pos: torch.Tensor


def verify_inputs(B: int, L: int, Hq: int, Hkv: int, D: int, W: int, *, seed: int = 0,
                  dtype: torch.dtype = torch.bfloat16, device="cpu", pos_lo: int = 128,
                  pos_hi: int = 262144) -> VerifyInputs:
    """Draw verify inputs: L drafted tokens per sequence and a full W-slot ring."""
    g = _gen(seed, device)
    f32 = torch.float32
    q = torch.randn(B, L, Hq, D, generator=g, device=device, dtype=f32)
    k_new = torch.randn(B, L, Hkv, D, generator=g, device=device, dtype=f32)
    v_new = torch.randn(B, L, Hkv, D, generator=g, device=device, dtype=f32)
    k_ring = torch.randn(B, Hkv, W, D, generator=g, device=device, dtype=f32)
    v_ring = torch.randn(B, Hkv, W, D, generator=g, device=device, dtype=f32)
    sink = torch.randn(Hq, generator=g, device=device, dtype=f32)
    pos = torch.randint(pos_lo, pos_hi, (B,), generator=g, device=device, dtype=torch.int64)
    return VerifyInputs(q.to(dtype), k_new.to(dtype), v_new.to(dtype), k_ring.to(dtype),
                        v_ring.to(dtype), sink, pos)


def ring_from_history(k_hist: torch.Tensor, v_hist: torch.Tensor, pos: torch.Tensor, W: int):
    """Lay a full key/value history ``[B,T,Hkv,D]`` into W-slot rings ``[B,Hkv,W,D]``.

    Slot s of sequence b holds the latest position p <= pos[b] with p % W == s;
    slots whose position would be negative are zero.  This is pure data
    movement (the cache layout), used by tests to build a ring whose contents
    are known from a history.
    """
    B, T, Hkv, D = k_hist.shape
    kr = torch.zeros(B, Hkv, W, D, dtype=k_hist.dtype, device=k_hist.device)
    vr = torch.zeros_like(kr)
    for b in range(B):
        p_now = int(pos[b])
        for s in range(W):
            p = p_now - ((p_now - s) % W)
            if p >= 0:
                kr[b, :, s] = k_hist[b, p]
                vr[b, :, s] = v_hist[b, p]
    return kr, vr
