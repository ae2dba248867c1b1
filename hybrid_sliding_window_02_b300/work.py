"""Algorithmic work accounting (FLOPs and bytes) for the attention calls.

Only in-window (query, key) pairs count: masked tile work and the dense T^2
that the window avoids are not work.  A pair costs 2*D FLOPs for the score and
2*D for the value accumulation.  Bytes count every input read once and every
output written once.
"""
from __future__ import annotations


def window_pairs(T: int, W: int) -> int:
    """Number of (i, j) with 0 <= j <= i < T and i - j < W: sum_i min(i+1, W)."""
    if T <= 0:
        return 0
    if W >= T:
        return T * (T + 1) // 2
    return W * (W + 1) // 2 + (T - W) * W


def prefill_flops(B: int, T: int, Hq: int, D: int, W: int) -> int:
    return 4 * D * B * Hq * window_pairs(T, W)


def prefill_bytes(B: int, T: int, Hq: int, Hkv: int, D: int, in_bytes: int,
                  out_bytes: int = 4, with_lse: bool = True) -> int:
    rd = B * T * (Hq + 2 * Hkv) * D * in_bytes + Hq * 4
    wr = B * T * Hq * D * out_bytes + (B * Hq * T * 4 if with_lse else 0)
    return rd + wr


def decode_flops(B: int, Hq: int, D: int, W: int) -> int:
    return 4 * D * B * Hq * W


def decode_bytes(B: int, Hq: int, Hkv: int, D: int, W: int, in_bytes: int,
                 with_lse: bool = True) -> int:
    rd = B * Hq * D * in_bytes + 2 * B * Hkv * W * D * in_bytes + B * 8 + Hq * 4
    wr = B * Hq * D * 4 + (B * Hq * 4 if with_lse else 0)
    return rd + wr


def append_bytes(B: int, Hkv: int, D: int, in_bytes: int) -> int:
    """Ring append: the new token's k and v read, written into one ring slot
    per (sequence, kv head); pos read."""
    return 2 * (2 * B * Hkv * D * in_bytes) + B * 8


def rope_bytes(B: int, T: int, H: int, D: int, in_bytes: int) -> int:
    """RoPE in place on x [B, T, H, D]: x read and written once; pos0 read."""
    return 2 * B * T * H * D * in_bytes + B * 8


def rope_append_bytes(B: int, Hq: int, Hkv: int, D: int, in_bytes: int) -> int:
    """Fused rotate-and-append: the ring append plus the new token's q read and
    its rotated copy written."""
    return append_bytes(B, Hkv, D, in_bytes) + 2 * B * Hq * D * in_bytes


def verify_pairs(L: int, W: int, pos: int) -> int:
    """(query, key) pairs of one verify group row set: drafted token j at
    position pos + j sees min(pos + j + 1, W) keys."""
    return sum(min(pos + j + 1, W) for j in range(L))


def verify_flops(B: int, L: int, Hq: int, D: int, W: int) -> int:
    """FLOPs of a verify call with every window full (pos >= W - 1)."""
    return 4 * D * B * Hq * L * W


def verify_bytes(B: int, L: int, Hq: int, Hkv: int, D: int, W: int, in_bytes: int,
                 with_lse: bool = True) -> int:
    rd = (B * L * Hq * D * in_bytes + 2 * B * L * Hkv * D * in_bytes
          + 2 * B * Hkv * W * D * in_bytes + B * 8 + Hq * 4)
    wr = B * L * Hq * D * 4 + (B * Hq * L * 4 if with_lse else 0)
    return rd + wr


def hybrid_reduction(T: int, W: int = 128, n_swa: int = 5, n_ga: int = 1):
    """(attention-FLOP ratio, KV-cache ratio) of an all-global stack over a
    hybrid stack with n_swa window layers per n_ga global layers, at length T.

    The MiMo-V2-Flash pages state "about 6x" for 5:1 with W = 128 ("MiMo-V2-Flash
    Technical Report" summary, 核心方法; "wiki-for-amaranth" notes, 关键架构决策).
    """
    n = n_swa + n_ga
    flop = n * window_pairs(T, T) / (n_swa * window_pairs(T, W) + n_ga * window_pairs(T, T))
    kv = n * T / (n_swa * min(W, T) + n_ga * T)
    return flop, kv
