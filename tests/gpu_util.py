"""Helpers for the GPU parity tests: move seeded inputs to the device, call the
CUDA library through its C-ABI binding, and measure errors against the
oracle.  Holds none of the method's arithmetic."""
from __future__ import annotations

import numpy as np
import torch

import gated_deltanet_linear_pre_gb300 as gdn

# tolerances of the parity contract (max |x - ref| / max |ref| per tensor)
TOL_F16 = 2e-3      # fp16 outputs
TOL_F32 = 1e-4      # fp32 outputs and the final fp32 state
TOL_STAGE = 1e-5    # fp32 stage tensors of gdn_pre (no accumulation involved)
# The same metric per (sequence, head) slice is stricter than the contract's per-tensor one: the split
# bf16 products' absolute error scales with their operands, not with the slice's own largest output,
# so a head whose outputs are small next to the tensor's largest value shows a larger ratio.  Slices
# are held to 5x the per-tensor bars.
TOL_SLICE_F32 = 5e-4
TOL_SLICE_F16 = 1e-2


def max_rel(x, ref) -> float:
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert x.shape == ref.shape, (x.shape, ref.shape)
    if ref.size == 0:
        return 0.0
    den = np.abs(ref).max()
    err = np.abs(x - ref).max()
    return float(err / den) if den > 0 else float(err)


def max_rel_slices(x, ref, cu_seqlens=None, token_axis=0, head_axis=1):
    """The same metric per (sequence, head) slice, the worst slice returned: each slice is held to its
    own max |ref|, so a head or sequence with a small output or state is not judged against the
    tensor's largest value.  With cu_seqlens the token axis is cut into sequences; without it the
    token axis indexes sequences already (a state tensor [n_seq, hv, ...])."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert x.shape == ref.shape, (x.shape, ref.shape)
    n = ref.shape[token_axis]
    bounds = [(int(cu_seqlens[s]), int(cu_seqlens[s + 1])) for s in range(len(cu_seqlens) - 1)] \
        if cu_seqlens is not None else [(i, i + 1) for i in range(n)]
    worst = 0.0
    for lo, hi in bounds:
        if hi <= lo:
            continue
        xs = np.take(x, range(lo, hi), axis=token_axis)
        rs = np.take(ref, range(lo, hi), axis=token_axis)
        for h in range(ref.shape[head_axis]):
            worst = max(worst, max_rel(np.take(xs, h, axis=head_axis), np.take(rs, h, axis=head_axis)))
    return worst


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t if dtype is None else t.to(dtype)


def dims_of(inp):
    hk, hv, dk, dv = inp.dims
    return gdn.dims(hk, hv, dk, dv, 1e-6)


def device_inputs(inp):
    return dict(cu=dev(inp.cu_seqlens), qkv=dev(inp.qkv), conv_w=dev(inp.conv_w), hist=dev(inp.hist),
                a=dev(inp.a), b=dev(inp.b), A_log=dev(inp.A_log), dt_bias=dev(inp.dt_bias), z=dev(inp.z),
                gamma=dev(inp.gamma), S0=dev(inp.S0))


def run_layer(inp, out_f32=None, in_place_state=False):
    """gdn_layer on the device; returns numpy y, hist_out, S_out."""
    out_f32 = inp.out_f32 if out_f32 is None else out_f32
    d = dims_of(inp)
    x = device_inputs(inp)
    T, n_seq = inp.total_tokens, inp.n_seq
    hv, dv = d.hv, d.dv
    y = torch.empty((T, hv, dv), device="cuda", dtype=torch.float32 if out_f32 else torch.float16)
    hist_out = torch.empty_like(x["hist"])
    S_out = x["S0"] if in_place_state else torch.empty_like(x["S0"])
    ws = torch.empty(gdn.gdn_layer_workspace_bytes(d, n_seq, T), device="cuda", dtype=torch.uint8)
    gdn.gdn_layer(d, x["cu"], T, x["qkv"], x["conv_w"], x["hist"], hist_out, x["a"], x["b"], x["z"], x["A_log"],
                  x["dt_bias"], x["gamma"], x["S0"], S_out, out_f32, y, ws)
    torch.cuda.synchronize()
    return dict(y=y.float().cpu().numpy(), hist_out=hist_out.cpu().numpy(), S_out=S_out.cpu().numpy())


def run_pre(inp):
    d = dims_of(inp)
    x = device_inputs(inp)
    T = inp.total_tokens
    hk, hv, dk, dv = inp.dims
    f32 = dict(device="cuda", dtype=torch.float32)
    out = dict(q=torch.empty((T, hk, dk), **f32), k=torch.empty((T, hk, dk), **f32),
               v=torch.empty((T, hv, dv), **f32), lam=torch.empty((T, hv), **f32),
               beta=torch.empty((T, hv), **f32), hist_out=torch.empty_like(x["hist"]))
    gdn.gdn_pre(d, x["cu"], T, x["qkv"], x["conv_w"], x["hist"], out["hist_out"], x["a"], x["b"], x["A_log"],
                x["dt_bias"], out["q"], out["k"], out["v"], out["lam"], out["beta"])
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def run_scan(d, cu_seqlens, q, k, v, lam, beta, S0, in_place=False):
    """gdn_scan on fp32 copies of the given arrays; returns numpy o, S_out."""
    T = q.shape[0]
    f = torch.float32
    S_in = dev(S0, f)
    S_out = S_in if in_place else torch.empty_like(S_in)
    o = torch.empty((T, d.hv, d.dv), device="cuda", dtype=f)
    nbytes = gdn.gdn_scan_workspace_bytes(d, len(cu_seqlens) - 1, T)
    ws = torch.empty(nbytes, device="cuda", dtype=torch.uint8) if nbytes else None
    gdn.gdn_scan(d, dev(np.asarray(cu_seqlens, np.int32)), T, dev(q, f), dev(k, f), dev(v, f), dev(lam, f),
                 dev(beta, f), S_in, S_out, o, ws)
    torch.cuda.synchronize()
    return o.cpu().numpy(), S_out.cpu().numpy()


def run_post(d, o, z, gamma, out_f32):
    T = o.shape[0]
    y = torch.empty(o.shape, device="cuda", dtype=torch.float32 if out_f32 else torch.float16)
    gdn.gdn_post(d, T, dev(o, torch.float32), dev(z), dev(gamma), out_f32, y)
    torch.cuda.synchronize()
    return y.float().cpu().numpy()
