"""Seeded synthetic inputs for the GDN prompt-prefill path.

This module only draws random numbers; it holds none of the method's
arithmetic.  Both the CUDA path's tests/benchmark and the CPU oracle take
their inputs from here.

Recipe (shapes and distributions of the pages' production layer: hk=16 key
heads, hv=48 value heads, dk=dv=128, 10240 packed q|k|v channels):

  draw order, one ``numpy.random.Generator(PCG64(seed))`` per layer:
    lengths (varlen batches only), qkv, conv_w, hist, a, b, A_log, dt_bias,
    z, gamma, S0
  qkv      fp16 [T, C]            N(0, 1)
  conv_w   fp32 [C, 4]            N(0, 0.25)   (second argument = std)
  hist     fp16 [n_seq, C, 3]     zeros, or N(0, 1) when seeded nonzero
  a, b     fp16 [T, hv]           N(0, 1)
  A_log    fp32 [hv]              log U(1, 16)   (or log U(lo, hi) if given)
  dt_bias  fp32 [hv]              N(0, 0.1)
  z        fp16 [T, hv, dv]       N(0, 1)
  gamma    fp32 [dv]              1 + 0.1 N(0, 1)
  S0       fp32 [n_seq, hv, dk, dv]  zeros, or N(0, S0_std)
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

HK, HV, DK, DV = 16, 48, 128, 128
BASE_SEED = 21


def channels(hk: int = HK, hv: int = HV, dk: int = DK, dv: int = DV) -> int:
    return 2 * hk * dk + hv * dv


@dataclass
class LayerInputs:
    qkv: np.ndarray         # fp16 [T, C]
    conv_w: np.ndarray      # fp32 [C, 4]
    hist: np.ndarray        # fp16 [n_seq, C, 3], oldest token first
    a: np.ndarray           # fp16 [T, hv]
    b: np.ndarray           # fp16 [T, hv]
    A_log: np.ndarray       # fp32 [hv]
    dt_bias: np.ndarray     # fp32 [hv]
    z: np.ndarray           # fp16 [T, hv, dv]
    gamma: np.ndarray       # fp32 [dv]
    S0: np.ndarray          # fp32 [n_seq, hv, dk, dv]
    cu_seqlens: np.ndarray  # int32 [n_seq + 1]
    out_f32: bool = False
    dims: tuple = field(default=(HK, HV, DK, DV))

    @property
    def n_seq(self) -> int:
        return int(self.cu_seqlens.size - 1)

    @property
    def total_tokens(self) -> int:
        return int(self.cu_seqlens[-1])


def _normal(rng, shape, std, dtype):
    return (rng.standard_normal(shape, dtype=np.float32) * np.float32(std)).astype(dtype)


def make_layer(seed: int, lengths=None, *, n_seq_random: int = 0, max_len: int = 4096,
               hist_nonzero: bool = False, S0_std: float = 0.0, A_log_range=(1.0, 16.0),
               out_f32: bool = False, dims=(HK, HV, DK, DV)) -> LayerInputs:
    """One layer's inputs.  Either ``lengths`` (list of sequence lengths) or
    ``n_seq_random`` sequences with lengths uniform in [1, max_len]."""
    hk, hv, dk, dv = dims
    C = channels(hk, hv, dk, dv)
    rng = np.random.Generator(np.random.PCG64(seed))
    if lengths is None:
        lengths = rng.integers(1, max_len + 1, size=n_seq_random)
    lengths = np.asarray(lengths, dtype=np.int64)
    cu = np.zeros(lengths.size + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lengths)
    T = int(cu[-1])
    n_seq = lengths.size
    qkv = _normal(rng, (T, C), 1.0, np.float16)
    conv_w = _normal(rng, (C, 4), 0.25, np.float32)
    if hist_nonzero:
        hist = _normal(rng, (n_seq, C, 3), 1.0, np.float16)
    else:
        hist = np.zeros((n_seq, C, 3), dtype=np.float16)
    a = _normal(rng, (T, hv), 1.0, np.float16)
    b = _normal(rng, (T, hv), 1.0, np.float16)
    lo, hi = A_log_range
    A_log = np.log(rng.uniform(lo, hi, size=hv)).astype(np.float32)
    dt_bias = _normal(rng, (hv,), 0.1, np.float32)
    z = _normal(rng, (T, hv, dv), 1.0, np.float16)
    gamma = (1.0 + 0.1 * rng.standard_normal(dv)).astype(np.float32)
    if S0_std > 0:
        S0 = _normal(rng, (n_seq, hv, dk, dv), S0_std, np.float32)
    else:
        S0 = np.zeros((n_seq, hv, dk, dv), dtype=np.float32)
    return LayerInputs(qkv=qkv, conv_w=conv_w, hist=hist, a=a, b=b, A_log=A_log,
                       dt_bias=dt_bias, z=z, gamma=gamma, S0=S0, cu_seqlens=cu,
                       out_f32=out_f32, dims=tuple(dims))


# ---- the five workloads -----------------------------------------------------
def single_layer_t37() -> LayerInputs:
    """One sequence of 37 tokens, zero history and state, fp16 output."""
    return make_layer(BASE_SEED, [37])


def single_layer_boundary(T: int, out_f32: bool) -> LayerInputs:
    """T in {1, 3, 300, 512}: seeded nonzero history and S0 ~ N(0, 0.02)."""
    return make_layer(BASE_SEED, [T], hist_nonzero=True, S0_std=0.02, out_f32=out_f32)


def stack_layer(layer: int, T: int = 2048, out_f32: bool = False) -> LayerInputs:
    """Layer ``layer`` of the 36-layer T=2048 stack (seed 21 + layer)."""
    return make_layer(BASE_SEED + layer, [T], out_f32=out_f32)


def varlen_batch(n_seq: int = 8, max_len: int = 4096, out_f32: bool = False) -> LayerInputs:
    """8 sequences, lengths uniform in [1, 4096], own history and S0 each."""
    return make_layer(BASE_SEED, None, n_seq_random=n_seq, max_len=max_len, hist_nonzero=True,
                      S0_std=0.02, out_f32=out_f32)


def long_prompt(T: int = 32768, out_f32: bool = False) -> LayerInputs:
    """One long sequence with decays near 1: A_log = log U(0.01, 0.1)."""
    return make_layer(BASE_SEED, [T], A_log_range=(0.01, 0.1), out_f32=out_f32)


def decode_batch(n_seq: int = 256, layer: int = 0, out_f32: bool = False) -> LayerInputs:
    """One decode step for n_seq sequences: one token each, carried history and
    state from earlier tokens (nonzero history, S0 ~ N(0, 0.02))."""
    return make_layer(BASE_SEED + 1000 + layer, [1] * n_seq, hist_nonzero=True, S0_std=0.02, out_f32=out_f32)
