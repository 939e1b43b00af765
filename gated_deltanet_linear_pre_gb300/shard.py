"""Head sharding of one GDN prefill layer across ranks.

Every stage of the layer is local to a key head and its value heads: the
depthwise conv and SiLU act per channel, the L2 norm per q/k head, the
recurrence per value head (reading its key head's q and k), the gated RMSNorm
per (token, value head).  Rank r of W therefore takes key heads
[r hk/W, (r+1) hk/W) with their value heads [r hv/W, (r+1) hv/W) and runs the
whole layer on them with no data exchanged; only a consumer that wants full
rows needs the outputs gathered across ranks (``gather_outputs``).
("Round 30 Track C Audit: gdn_pre, gdn_post, and gdn_scanr_4", section 1: the
kernels reduce over one head at a time -- the per-key-head q/k sums of squares,
the per-head output reduction of gdn_post -- and the scan works head by head.)

This module only slices and reassembles arrays (numpy arrays or torch tensors,
any device); it holds none of the method's arithmetic.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class HeadShard:
    rank: int
    world: int
    j0: int  # first key head
    j1: int  # one past the last key head
    h0: int  # first value head
    h1: int  # one past the last value head

    @property
    def hk(self) -> int:
        return self.j1 - self.j0

    @property
    def hv(self) -> int:
        return self.h1 - self.h0


def head_shard(hk: int, hv: int, world: int, rank: int) -> HeadShard:
    """Rank `rank`'s key heads and their value heads (value head h reads key head h / (hv / hk))."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside a world of {world}")
    if hk % world != 0 or hv % hk != 0:
        raise ValueError(f"hk={hk} must split evenly over {world} ranks and hv={hv} be a multiple of hk")
    per_rank = hk // world
    group = hv // hk
    j0 = rank * per_rank
    return HeadShard(rank, world, j0, j0 + per_rank, j0 * group, (j0 + per_rank) * group)


def channel_index(sh: HeadShard, hk: int, hv: int, dk: int = 128, dv: int = 128) -> np.ndarray:
    """Positions, in the packed q | k | v channel order, of the shard's channels, in the same order
    (its q heads, then its k heads, then its v heads), so that the slice is itself a packed layer."""
    q = np.arange(sh.j0 * dk, sh.j1 * dk)
    k = hk * dk + np.arange(sh.j0 * dk, sh.j1 * dk)
    v = 2 * hk * dk + np.arange(sh.h0 * dv, sh.h1 * dv)
    return np.concatenate([q, k, v])


def _take(x, idx, axis):
    """x indexed by `idx` along `axis` (numpy or torch, contiguous result)."""
    if isinstance(x, np.ndarray):
        return np.ascontiguousarray(np.take(x, idx, axis=axis))
    import torch
    return torch.index_select(x, axis, torch.as_tensor(idx, device=x.device)).contiguous()


def shard_layer_inputs(x: dict, sh: HeadShard, hk: int, hv: int, dk: int = 128, dv: int = 128) -> dict:
    """The shard's part of one layer's inputs.  `x` holds qkv [T, C], conv_w [C, 4], hist [n_seq, C, 3],
    a and b [T, hv], A_log and dt_bias [hv], z [T, hv, dv], gamma [dv], S0 [n_seq, hv, dk, dv]; other keys
    (cu_seqlens, ...) pass through."""
    ch = channel_index(sh, hk, hv, dk, dv)
    heads = np.arange(sh.h0, sh.h1)
    out = dict(x)
    out["qkv"] = _take(x["qkv"], ch, 1)
    out["conv_w"] = _take(x["conv_w"], ch, 0)
    out["hist"] = _take(x["hist"], ch, 1)
    for key in ("a", "b", "z", "S0"):
        out[key] = _take(x[key], heads, 1)
    for key in ("A_log", "dt_bias"):
        out[key] = _take(x[key], heads, 0)
    return out


def gather_outputs(parts: list, hk: int, hv: int, dk: int = 128, dv: int = 128) -> dict:
    """Full-width outputs from every rank's shard outputs (dicts with y [T, hv/W, dv], hist_out
    [n_seq, C/W, 3] and S_out [n_seq, hv/W, dk, dv]), in rank order."""
    world = len(parts)
    shards = [head_shard(hk, hv, world, r) for r in range(world)]
    first = parts[0]
    numpy = isinstance(first["y"], np.ndarray)
    if numpy:
        cat = lambda xs, axis: np.concatenate(xs, axis=axis)
    else:
        import torch
        cat = lambda xs, axis: torch.cat(xs, dim=axis)
    y = cat([p["y"] for p in parts], 1)
    S_out = cat([p["S_out"] for p in parts], 1)
    # history channels go back to their packed positions
    ch = np.concatenate([channel_index(sh, hk, hv, dk, dv) for sh in shards])
    order = np.argsort(ch)
    hist = cat([p["hist_out"] for p in parts], 1)
    hist = _take(hist, order, 1)
    return {"y": y, "hist_out": hist, "S_out": S_out}
