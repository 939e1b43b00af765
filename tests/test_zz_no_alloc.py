"""gdn_scan_noalloc: the scan for callers that cannot allocate device memory.

Some callers have no way to hand the library a device workspace: a host
program that uses the plain C ABI with no allocator of its own, or a service
that forbids device allocation once it is running.  gdn_scan_noalloc serves
them with a fixed scratch array that the library owns.  This test calls it
through the C ABI twice in a row and checks both results against gdn_scan
with an ordinary workspace, within the fp32 tolerance of the parity tests.
It lives in a file that pytest collects last.
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


def _stage_tensors(inp):
    ref = oracle.layer(inp, heads=[0])
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(np.asarray(a, np.float32))).cuda()
    return [dev(ref[k]) for k in ("q", "k", "v", "lam", "beta")]


def test_noalloc_scan_matches_workspace_scan_twice():
    import gpu_util as u
    import gated_deltanet_linear_pre_gb300 as gdn
    inp = gin.make_layer(77, [130, 0, 200], hist_nonzero=True, S0_std=0.02)
    d = u.dims_of(inp)
    T, n_seq = inp.total_tokens, inp.n_seq
    assert gdn.gdn_scan_workspace_bytes(d, n_seq, T) <= (64 << 20)
    q, k, v, lam, beta = _stage_tensors(inp)
    cu = u.dev(inp.cu_seqlens)
    S_in = u.dev(inp.S0, torch.float32)

    o_ref = torch.empty_like(v)
    S_ref = torch.empty_like(S_in)
    ws = torch.empty(gdn.gdn_scan_workspace_bytes(d, n_seq, T), device="cuda", dtype=torch.uint8)
    gdn.gdn_scan(d, cu, T, q, k, v, lam, beta, S_in, S_ref, o_ref, ws)
    torch.cuda.synchronize()
    o_ref, S_ref = o_ref.cpu().numpy(), S_ref.cpu().numpy()

    for _ in range(2):  # the shared scratch keeps the previous call's contents
        o = torch.full_like(v, float("nan"))
        S_out = torch.full_like(S_in, float("nan"))
        gdn.gdn_scan_noalloc(d, cu, T, q, k, v, lam, beta, S_in, S_out, o)
        gdn.gdn_scan_noalloc_check()  # no bounded wait of the scan ran out (synchronises)
        torch.cuda.synchronize()
        assert u.max_rel(o.cpu().numpy(), o_ref) <= u.TOL_F32
        assert u.max_rel(S_out.cpu().numpy(), S_ref) <= u.TOL_F32


def test_noalloc_scan_rejects_batches_beyond_its_scratch():
    import gated_deltanet_linear_pre_gb300 as gdn
    d = gdn.dims()
    T = 32768
    assert gdn.gdn_scan_workspace_bytes(d, 1, T) > (64 << 20)
    f = lambda *s: torch.empty(*s, device="cuda", dtype=torch.float32)
    cu = torch.tensor([0, T], dtype=torch.int32, device="cuda")
    with pytest.raises(gdn.GdnError) as ei:
        gdn.gdn_scan_noalloc(d, cu, T, f(T, 16, 128), f(T, 16, 128), f(T, 48, 128), f(T, 48), f(T, 48),
                             f(1, 48, 128, 128), f(1, 48, 128, 128), f(T, 48, 128))
    assert ei.value.status == 2 and "maximum" in str(ei.value)
