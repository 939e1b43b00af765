"""Failure detection on the GPU without a fault: every wait inside the scan
kernels is bounded, and an expired wait is reported to the host.

The self-test entry point withholds one operand copy of the recurrence
kernel, so that a bounded wait in each of its CTAs runs out (about two
seconds); the kernel records the failure in the workspace, releases what it
holds and stops.  gdn_scan_check then reports GDN_ERR_TIMEOUT, and the same
context goes on to compute a correct scan.
"""
import numpy as np
import pytest

import oracle
from gated_deltanet_linear_pre_gb300 import inputs as gin

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_deltanet_linear_pre_gb300 import build
    build.build()


def _scan_args(inp):
    import gpu_util as u
    import gated_deltanet_linear_pre_gb300 as gdn
    ref = oracle.layer(inp)
    d = u.dims_of(inp)
    T, n_seq = inp.total_tokens, inp.n_seq
    f = torch.float32
    args = dict(cu=u.dev(inp.cu_seqlens), q=u.dev(ref["q"], f), k=u.dev(ref["k"], f), v=u.dev(ref["v"], f),
                lam=u.dev(ref["lam"], f), beta=u.dev(ref["beta"], f), S_in=u.dev(inp.S0, f))
    ws = torch.empty(gdn.gdn_scan_workspace_bytes(d, n_seq, T), device="cuda", dtype=torch.uint8)
    return ref, d, T, args, ws


def test_scan_check_reports_ok_after_normal_runs():
    import gpu_util as u
    import gated_deltanet_linear_pre_gb300 as gdn
    inp = gin.make_layer(90, [150, 70], hist_nonzero=True, S0_std=0.02)
    ref, d, T, a, ws = _scan_args(inp)
    o = torch.empty((T, d.hv, d.dv), device="cuda")
    S_out = torch.empty_like(a["S_in"])
    gdn.gdn_scan(d, a["cu"], T, a["q"], a["k"], a["v"], a["lam"], a["beta"], a["S_in"], S_out, o, ws)
    gdn.gdn_scan_check(ws)
    # and through gdn_layer's workspace
    x = u.device_inputs(inp)
    lws = torch.empty(gdn.gdn_layer_workspace_bytes(d, inp.n_seq, T), device="cuda", dtype=torch.uint8)
    y = torch.empty((T, d.hv, d.dv), device="cuda", dtype=torch.float16)
    gdn.gdn_layer(d, x["cu"], T, x["qkv"], x["conv_w"], x["hist"], torch.empty_like(x["hist"]), x["a"], x["b"],
                  x["z"], x["A_log"], x["dt_bias"], x["gamma"], x["S0"], torch.empty_like(x["S0"]), False, y, lws)
    gdn.gdn_layer_check(d, inp.n_seq, T, lws)
    # and no fault that would leave the context unusable was seen (a non-synchronising check)
    gdn.gdn_last_async_error()


def test_expired_wait_is_reported_and_the_context_stays_usable():
    import gpu_util as u
    import gated_deltanet_linear_pre_gb300 as gdn
    inp = gin.make_layer(91, [300], hist_nonzero=True, S0_std=0.02)
    ref, d, T, a, ws = _scan_args(inp)
    o = torch.empty((T, d.hv, d.dv), device="cuda")
    S_out = torch.empty_like(a["S_in"])
    gdn.gdn_scan_selftest_timeout(d, a["cu"], T, a["q"], a["k"], a["v"], a["lam"], a["beta"], a["S_in"], S_out,
                                  o, ws)
    with pytest.raises(gdn.GdnError) as ei:
        gdn.gdn_scan_check(ws)
    assert ei.value.status == 6 and "expired" in str(ei.value)
    # the same context, workspace and buffers: a normal scan is correct and reports OK
    gdn.gdn_scan(d, a["cu"], T, a["q"], a["k"], a["v"], a["lam"], a["beta"], a["S_in"], S_out, o, ws)
    gdn.gdn_scan_check(ws)
    assert u.max_rel(o.cpu().numpy(), ref["o"]) <= u.TOL_F32
    assert u.max_rel(S_out.cpu().numpy(), ref["S_out"]) <= u.TOL_F32


def test_expired_wait_across_kernels_is_reported():
    """The recurrence kernel waits, bounded, on the prep kernel's per-(chunk, value head) ready flags.
    With one flag left unset (chunk slot 1, value head 0) that wait runs out in the CTAs of head 0:
    the check reports GDN_ERR_TIMEOUT, and the same context then computes a correct scan."""
    import gpu_util as u
    import gated_deltanet_linear_pre_gb300 as gdn
    inp = gin.make_layer(93, [200], hist_nonzero=True, S0_std=0.02)
    ref, d, T, a, ws = _scan_args(inp)
    o = torch.empty((T, d.hv, d.dv), device="cuda")
    S_out = torch.empty_like(a["S_in"])
    gdn.gdn_scan_selftest_withhold_flag(d, a["cu"], T, a["q"], a["k"], a["v"], a["lam"], a["beta"], a["S_in"],
                                        S_out, o, ws)
    with pytest.raises(gdn.GdnError) as ei:
        gdn.gdn_scan_check(ws)
    assert ei.value.status == 6
    gdn.gdn_last_async_error()  # an expired wait is reported, not a fault: the context is intact
    gdn.gdn_scan(d, a["cu"], T, a["q"], a["k"], a["v"], a["lam"], a["beta"], a["S_in"], S_out, o, ws)
    gdn.gdn_scan_check(ws)
    assert u.max_rel(o.cpu().numpy(), ref["o"]) <= u.TOL_F32
    assert u.max_rel(S_out.cpu().numpy(), ref["S_out"]) <= u.TOL_F32


@pytest.mark.parametrize("lens", [[2048], [1000, 700, 350]])
def test_prep_fallback_alone_gives_the_same_scan(lens):
    """With no SM kept for prep after its first round, the one CTA the fallback keeps takes every
    remaining task; the scan must come out bit for bit as the normal one."""
    import gpu_util as u
    import gated_deltanet_linear_pre_gb300 as gdn
    inp = gin.make_layer(92, lens, hist_nonzero=True, S0_std=0.02)
    d = u.dims_of(inp)
    T, n_seq = inp.total_tokens, inp.n_seq
    x = u.device_inputs(inp)
    f = dict(device="cuda", dtype=torch.float32)
    q, k = torch.empty((T, d.hk, d.dk), **f), torch.empty((T, d.hk, d.dk), **f)
    v, lam, beta = torch.empty((T, d.hv, d.dv), **f), torch.empty((T, d.hv), **f), torch.empty((T, d.hv), **f)
    gdn.gdn_pre(d, x["cu"], T, x["qkv"], x["conv_w"], x["hist"], torch.empty_like(x["hist"]), x["a"], x["b"],
                x["A_log"], x["dt_bias"], q, k, v, lam, beta)
    ws = torch.empty(gdn.gdn_scan_workspace_bytes(d, n_seq, T), device="cuda", dtype=torch.uint8)
    o1, o2 = torch.empty((T, d.hv, d.dv), **f), torch.empty((T, d.hv, d.dv), **f)
    S1, S2 = torch.empty_like(x["S0"]), torch.empty_like(x["S0"])
    gdn.gdn_scan(d, x["cu"], T, q, k, v, lam, beta, x["S0"], S1, o1, ws)
    gdn.gdn_scan_check(ws)
    gdn.gdn_scan_selftest_one_taker(d, x["cu"], T, q, k, v, lam, beta, x["S0"], S2, o2, ws)
    gdn.gdn_scan_check(ws)
    assert torch.equal(o1, o2) and torch.equal(S1, S2)
