"""GPU parity of gdn_step, the fused decode step (one token per sequence).

Reference: the fp64 oracle on a batch in which every sequence holds one token
(the decode step computes exactly that).  Bars as for the prefill path: fp16
outputs 2e-3, fp32 outputs and the final fp32 state 1e-4, history bit-exact.
A chain of decode steps must also reproduce a prefill of the same tokens.
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


def run_step(inp, out_f32=None, in_place_state=False, rows=None, hist=None, S0=None):
    """gdn_step on the device for the token rows `rows` of each sequence (default: the whole
    one-token batch); returns numpy y, hist_out, S_out."""
    import gpu_util as u
    import gated_deltanet_linear_pre_gb300 as gdn
    out_f32 = inp.out_f32 if out_f32 is None else out_f32
    d = u.dims_of(inp)
    n = inp.n_seq
    rows = np.arange(n) if rows is None else np.asarray(rows)
    hv, dv = d.hv, d.dv
    x = dict(qkv=u.dev(inp.qkv[rows]), a=u.dev(inp.a[rows]), b=u.dev(inp.b[rows]), z=u.dev(inp.z[rows]),
             hist=u.dev(inp.hist if hist is None else hist), S0=u.dev(inp.S0 if S0 is None else S0),
             conv_w=u.dev(inp.conv_w), A_log=u.dev(inp.A_log), dt_bias=u.dev(inp.dt_bias), gamma=u.dev(inp.gamma))
    y = torch.full((n, hv, dv), float("nan"), device="cuda", dtype=torch.float32 if out_f32 else torch.float16)
    hist_out = torch.empty_like(x["hist"])
    S_out = x["S0"] if in_place_state else torch.full_like(x["S0"], float("nan"))
    gdn.gdn_step(d, n, x["qkv"], x["conv_w"], x["hist"], hist_out, x["a"], x["b"], x["z"], x["A_log"],
                 x["dt_bias"], x["gamma"], x["S0"], S_out, out_f32, y)
    torch.cuda.synchronize()
    return dict(y=y.float().cpu().numpy(), hist_out=hist_out.cpu().numpy(), S_out=S_out.cpu().numpy())


def _hist_bits(h64):
    h16 = h64.astype(np.float16)
    assert np.array_equal(h16.astype(np.float64), h64)  # copies of fp16 inputs
    return h16.view(np.uint16)


@pytest.mark.parametrize("out_f32", [False, True])
@pytest.mark.parametrize("n_seq", [1, 7, 300])
def test_step_matches_oracle(n_seq, out_f32):
    import gpu_util as u
    inp = gin.make_layer(40 + n_seq, [1] * n_seq, hist_nonzero=True, S0_std=0.02, out_f32=out_f32)
    ref = oracle.layer(inp)
    got = run_step(inp)
    assert u.max_rel(got["y"], ref["y"]) <= (u.TOL_F32 if out_f32 else u.TOL_F16)
    assert u.max_rel(got["S_out"], ref["S_out"]) <= u.TOL_F32
    np.testing.assert_array_equal(got["hist_out"].view(np.uint16), _hist_bits(ref["hist_out"]))


def test_step_in_place_state():
    inp = gin.make_layer(61, [1] * 5, hist_nonzero=True, S0_std=0.02)
    a = run_step(inp, in_place_state=True)
    b = run_step(inp)
    np.testing.assert_array_equal(a["S_out"], b["S_out"])
    np.testing.assert_array_equal(a["y"], b["y"])


def test_step_degenerate_gates():
    # g -> 0 (A_log large, a large), beta -> 1 and -> 0 (b = +-12): the state is replaced,
    # kept or cleared as the recurrence says
    import gpu_util as u
    inp = gin.make_layer(62, [1] * 6, hist_nonzero=True, S0_std=0.05, A_log_range=(200.0, 400.0))
    inp.a[:] = np.float16(8.0)
    inp.b[:3] = np.float16(12.0)
    inp.b[3:] = np.float16(-12.0)
    ref = oracle.layer(inp)
    got = run_step(inp)
    assert u.max_rel(got["y"], ref["y"]) <= u.TOL_F16
    assert u.max_rel(got["S_out"], ref["S_out"]) <= u.TOL_F32


def test_step_chain_equals_prefill():
    # 6 decode steps carried through the returned history and state reproduce a prefill of
    # the same 6 tokens per sequence (oracle), token by token
    import gpu_util as u
    L, n = 6, 4
    full = gin.make_layer(63, [L] * n, hist_nonzero=True, S0_std=0.02)
    ref = oracle.layer(full)
    hist, S = full.hist, full.S0
    for t in range(L):
        rows = full.cu_seqlens[:-1] + t
        step = gin.LayerInputs(qkv=full.qkv, conv_w=full.conv_w, hist=hist, a=full.a, b=full.b, A_log=full.A_log,
                               dt_bias=full.dt_bias, z=full.z, gamma=full.gamma, S0=S,
                               cu_seqlens=np.arange(n + 1, dtype=np.int32))
        got = run_step(step, rows=rows)
        assert u.max_rel(got["y"], ref["y"][rows]) <= u.TOL_F16, t
        hist, S = got["hist_out"], got["S_out"]
    np.testing.assert_array_equal(hist.view(np.uint16), _hist_bits(ref["hist_out"]))
    assert u.max_rel(S, ref["S_out"]) <= u.TOL_F32


def test_step_matches_layer_path():
    # the fused step and gdn_layer on the same one-token batch agree within the fp32 bar
    import gpu_util as u
    inp = gin.make_layer(64, [1] * 33, hist_nonzero=True, S0_std=0.02, out_f32=True)
    a = run_step(inp)
    b = u.run_layer(inp)
    assert u.max_rel(a["y"], b["y"]) <= u.TOL_F32
    assert u.max_rel(a["S_out"], b["S_out"]) <= u.TOL_F32
    np.testing.assert_array_equal(a["hist_out"], b["hist_out"])


def test_step_empty_batch_is_a_no_op():
    import gpu_util as u
    import gated_deltanet_linear_pre_gb300 as gdn
    inp = gin.make_layer(65, [1], hist_nonzero=True)
    d = u.dims_of(inp)
    e16 = lambda *s: torch.empty(*s, device="cuda", dtype=torch.float16)
    e32 = lambda *s: torch.empty(*s, device="cuda", dtype=torch.float32)
    C = inp.qkv.shape[1]
    gdn.gdn_step(d, 0, e16(0, C), u.dev(inp.conv_w), e16(0, C, 3), e16(0, C, 3), e16(0, 48), e16(0, 48),
                 e16(0, 48, 128), u.dev(inp.A_log), u.dev(inp.dt_bias), u.dev(inp.gamma), e32(0, 48, 128, 128),
                 e32(0, 48, 128, 128), False, e16(0, 48, 128))
    torch.cuda.synchronize()


@pytest.mark.parametrize("hk,hv", [(2, 2), (4, 8), (2, 8)])
def test_step_other_head_counts(hk, hv):
    import gpu_util as u
    inp = gin.make_layer(80 + hk * 10 + hv, [1] * 9, hist_nonzero=True, S0_std=0.02, dims=(hk, hv, 128, 128))
    ref = oracle.layer(inp, hk=hk, hv=hv)
    got = run_step(inp)
    assert u.max_rel(got["y"], ref["y"]) <= u.TOL_F16
    assert u.max_rel(got["S_out"], ref["S_out"]) <= u.TOL_F32
    np.testing.assert_array_equal(got["hist_out"].view(np.uint16), _hist_bits(ref["hist_out"]))
