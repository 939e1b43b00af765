"""The scan and the layer replayed from captured CUDA graphs.

A captured graph freezes every launch argument, so nothing per call may come
from the host: the scan's per-chunk ready flags are tagged with a call count
the scan itself advances on the device.  Replays with new data in the static
input buffers must give exactly what direct calls give (the path is
deterministic: every task computes the same values wherever it runs), replay
after replay.
"""
import numpy as np
import pytest

from gated_deltanet_linear_pre_gb300 import inputs as gin

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_deltanet_linear_pre_gb300 import build
    build.build()


def _stage(inp, d):
    """gdn_pre's outputs for one layer (direct call)."""
    import gpu_util as u
    import gated_deltanet_linear_pre_gb300 as gdn
    x = u.device_inputs(inp)
    T = inp.total_tokens
    f = dict(device="cuda", dtype=torch.float32)
    out = dict(q=torch.empty((T, d.hk, d.dk), **f), k=torch.empty((T, d.hk, d.dk), **f),
               v=torch.empty((T, d.hv, d.dv), **f), lam=torch.empty((T, d.hv), **f), beta=torch.empty((T, d.hv), **f))
    gdn.gdn_pre(d, x["cu"], T, x["qkv"], x["conv_w"], x["hist"], torch.empty_like(x["hist"]), x["a"], x["b"],
                x["A_log"], x["dt_bias"], out["q"], out["k"], out["v"], out["lam"], out["beta"])
    out["S0"], out["cu"] = x["S0"], x["cu"]
    return out


def test_scan_replayed_from_a_graph_matches_direct_calls():
    import gpu_util as u
    import gated_deltanet_linear_pre_gb300 as gdn
    A, B = gin.stack_layer(4), gin.make_layer(33, [2048], hist_nonzero=True, S0_std=0.02)
    d = u.dims_of(A)
    T = A.total_tokens
    sa, sb = _stage(A, d), _stage(B, d)
    static = {k: v.clone() for k, v in sa.items()}
    o, S = torch.empty((T, d.hv, d.dv), device="cuda"), torch.empty_like(sa["S0"])
    ws = torch.empty(gdn.gdn_scan_workspace_bytes(d, 1, T), device="cuda", dtype=torch.uint8)

    def scan(src, o_, S_):
        gdn.gdn_scan(d, src["cu"], T, src["q"], src["k"], src["v"], src["lam"], src["beta"], src["S0"], S_, o_, ws)

    ref = {}
    for name, src in (("A", sa), ("B", sb)):
        o_r, S_r = torch.empty_like(o), torch.empty_like(S)
        scan(src, o_r, S_r)
        ref[name] = (o_r, S_r)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        scan(static, o, S)  # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        scan(static, o, S)
    for name in ("A", "B", "A", "B"):
        src = sa if name == "A" else sb
        for k in ("q", "k", "v", "lam", "beta", "S0"):
            static[k].copy_(src[k])
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(o, ref[name][0]) and torch.equal(S, ref[name][1]), name
    gdn.gdn_scan_check(ws)


def test_layer_replayed_from_a_graph_matches_direct_calls():
    import gpu_util as u
    import gated_deltanet_linear_pre_gb300 as gdn
    A, B = gin.single_layer_boundary(512, False), gin.make_layer(34, [512], hist_nonzero=True, S0_std=0.02)
    d = u.dims_of(A)
    T = A.total_tokens
    xa, xb = u.device_inputs(A), u.device_inputs(B)
    static = {k: v.clone() for k, v in xa.items()}
    y = torch.empty((T, d.hv, d.dv), device="cuda", dtype=torch.float16)
    S, hist = torch.empty_like(xa["S0"]), torch.empty_like(xa["hist"])
    ws = torch.empty(gdn.gdn_layer_workspace_bytes(d, 1, T), device="cuda", dtype=torch.uint8)

    def layer(x, y_, S_, h_):
        gdn.gdn_layer(d, x["cu"], T, x["qkv"], x["conv_w"], x["hist"], h_, x["a"], x["b"], x["z"], x["A_log"],
                      x["dt_bias"], x["gamma"], x["S0"], S_, False, y_, ws)

    ref = {}
    for name, x in (("A", xa), ("B", xb)):
        r = (torch.empty_like(y), torch.empty_like(S), torch.empty_like(hist))
        layer(x, *r)
        ref[name] = r
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        layer(static, y, S, hist)
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        layer(static, y, S, hist)
    for name in ("B", "A", "B"):
        x = xa if name == "A" else xb
        for k in static:
            static[k].copy_(x[k])
        g.replay()
        torch.cuda.synchronize()
        for got, want in zip((y, S, hist), ref[name]):
            assert torch.equal(got, want), name
    gdn.gdn_layer_check(d, 1, T, ws)


def test_scan_ignores_what_the_workspace_held():
    """Every ready flag reading "written" on entry (the workspace filled with u64 ones) changes nothing:
    the scan clears its flags itself before prep publishes them."""
    import gpu_util as u
    import gated_deltanet_linear_pre_gb300 as gdn
    A = gin.make_layer(35, [700, 64, 1, 1283], hist_nonzero=True, S0_std=0.02)
    d = u.dims_of(A)
    T = A.total_tokens
    sa = _stage(A, d)
    nbytes = gdn.gdn_scan_workspace_bytes(d, A.n_seq, T)
    outs = []
    for fill in (0, 1):
        ws = torch.zeros(nbytes // 8 + 1, device="cuda", dtype=torch.int64).fill_(fill).view(torch.uint8)
        o = torch.empty((T, d.hv, d.dv), device="cuda")
        S = torch.empty_like(sa["S0"])
        gdn.gdn_scan(d, sa["cu"], T, sa["q"], sa["k"], sa["v"], sa["lam"], sa["beta"], sa["S0"], S, o, ws)
        torch.cuda.synchronize()
        gdn.gdn_scan_check(ws)
        outs.append((o, S))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    assert np.isfinite(outs[1][0].cpu().numpy()).all()


def test_back_to_back_batches_of_different_shapes_share_one_workspace():
    """Calls queued back to back on one workspace (sized for the largest) with different batch shapes:
    every call's counters, flags and images start from what the previous call left, and each result
    must equal the same call on a fresh workspace."""
    import gpu_util as u
    import gated_deltanet_linear_pre_gb300 as gdn
    batches = [gin.make_layer(36, [1500, 40, 700], hist_nonzero=True, S0_std=0.02),
               gin.stack_layer(5),
               gin.make_layer(37, [64] * 9 + [3], hist_nonzero=True, S0_std=0.02),
               gin.make_layer(38, [2047], hist_nonzero=True, S0_std=0.02)]
    dims = [u.dims_of(b) for b in batches]
    shared = torch.empty(max(gdn.gdn_layer_workspace_bytes(d, b.n_seq, b.total_tokens) for d, b in zip(dims, batches)),
                         device="cuda", dtype=torch.uint8)
    xs = [u.device_inputs(b) for b in batches]

    def run(i, ws):
        b, d, x = batches[i], dims[i], xs[i]
        y = torch.empty((b.total_tokens, d.hv, d.dv), device="cuda", dtype=torch.float16)
        S, hist = torch.empty_like(x["S0"]), torch.empty_like(x["hist"])
        gdn.gdn_layer(d, x["cu"], b.total_tokens, x["qkv"], x["conv_w"], x["hist"], hist, x["a"], x["b"], x["z"],
                      x["A_log"], x["dt_bias"], x["gamma"], x["S0"], S, False, y, ws)
        return y, S, hist

    queued = [run(i, shared) for i in range(len(batches))]  # no synchronisation between the calls
    torch.cuda.synchronize()
    for i in range(len(batches)):
        b, d = batches[i], dims[i]
        fresh = run(i, torch.empty(gdn.gdn_layer_workspace_bytes(d, b.n_seq, b.total_tokens), device="cuda",
                                   dtype=torch.uint8))
        torch.cuda.synchronize()
        for got, want in zip(queued[i], fresh):
            assert torch.equal(got, want), i
