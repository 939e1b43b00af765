"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every entry point that include/gdn.h declares, and rejects bad arguments on
the host before anything is launched."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")
TESTING_HEADER = os.path.join(ROOT, "include", "gdn_testing.h")


@pytest.fixture(scope="module")
def L():
    from gated_deltanet_linear_pre_gb300 import build
    build.build()
    from gated_deltanet_linear_pre_gb300 import _native
    return _native.lib()


def declared_symbols(path=HEADER):
    text = open(path).read()
    return sorted(set(re.findall(r"GDN_API\s+[\w\s\*]+?\b(gdn_\w+)\s*\(", text)))


def test_hooks_stay_out_of_the_product_header():
    # the self-test entry points are declared in gdn_testing.h only
    assert not [s for s in declared_symbols() if "selftest" in s]
    assert set(declared_symbols(TESTING_HEADER)) == {"gdn_scan_selftest_timeout", "gdn_scan_selftest_one_taker",
                                                     "gdn_scan_selftest_withhold_flag", "gdn_layer_selftest_stages"}


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for name in ("gdn_pre", "gdn_scan", "gdn_post", "gdn_layer", "gdn_step", "gdn_scan_workspace_bytes",
                 "gdn_layer_workspace_bytes", "gdn_status_string", "gdn_last_error_string",
                 "gdn_last_async_error", "gdn_scan_noalloc_check"):
        assert name in syms


def test_library_exports_every_declared_symbol(L):
    from gated_deltanet_linear_pre_gb300 import build
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT\s+(gdn_\w+)", out))
    declared = set(declared_symbols()) | set(declared_symbols(TESTING_HEADER))
    assert declared <= exported
    # nothing but the ABI and its declared test hooks is exported under the gdn_ prefix
    assert exported == declared
    for name in declared:
        assert hasattr(L, name)


def test_status_strings(L):
    names = [L.gdn_status_string(i).decode() for i in range(7)]
    assert names == ["GDN_OK", "GDN_ERR_INVALID_ARG", "GDN_ERR_UNSUPPORTED", "GDN_ERR_ALIGNMENT",
                     "GDN_ERR_WORKSPACE", "GDN_ERR_CUDA", "GDN_ERR_TIMEOUT"]


def test_header_compiles_as_c(tmp_path):
    src = tmp_path / "t.c"
    src.write_text('#include "gdn.h"\n#include "gdn_testing.h"\nint main(void){ gdn_dims d = {16,48,128,128,1e-6f};'
                   ' return (int)gdn_layer_workspace_bytes(&d, 1, 0) & 0; }\n')
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-c", "-I", os.path.join(ROOT, "include"), str(src),
                    "-o", str(tmp_path / "t.o")], check=True)


def test_workspace_sizes(L):
    from gated_deltanet_linear_pre_gb300 import _native as N
    d = N.dims()
    T = 2048
    ws = N.gdn_layer_workspace_bytes(d, 1, T)
    stage = T * (2 * 16 * 128 + 2 * 48 * 128 + 2 * 48) * 4
    assert ws >= stage
    assert ws % 256 == 0
    assert N.gdn_layer_workspace_bytes(d, 1, 0) >= 0


# ---- argument validation (host only: every call below fails before launch) ----
FAKE = 1 << 20  # a 16-byte-aligned address that is never dereferenced


def _pre(L, d, n_seq=1, T=4, **over):
    args = dict(cu=FAKE, qkv=FAKE, conv_w=FAKE, hist_in=FAKE, hist_out=2 * FAKE, a=FAKE, b=FAKE,
                A_log=FAKE, dt_bias=FAKE, qn=3 * FAKE, kn=4 * FAKE, vc=5 * FAKE, glog=6 * FAKE,
                beta=7 * FAKE)
    args.update(over)
    return L.gdn_pre(ctypes.byref(d) if d is not None else None, n_seq, T, *args.values(), None)


def test_pre_rejects_bad_arguments(L):
    from gated_deltanet_linear_pre_gb300 import _native as N
    assert _pre(L, None) == 1
    assert _pre(L, N.dims(dk=64)) == 2
    assert _pre(L, N.dims(hk=5, hv=48)) == 1
    assert _pre(L, N.dims(eps=0.0)) == 1
    assert _pre(L, N.dims(), n_seq=-1) == 1
    assert _pre(L, N.dims(), n_seq=0, T=3) == 1
    assert _pre(L, N.dims(), qkv=None) == 1
    assert _pre(L, N.dims(), qkv=FAKE + 8) == 3
    assert _pre(L, N.dims(), cu=None) == 1
    # outputs overlapping inputs or each other (hist_out == hist_in exactly is allowed: the in-place
    # history; a partial overlap is not)
    assert _pre(L, N.dims(), hist_in=2 * FAKE, hist_out=2 * FAKE + 16) == 1
    assert _pre(L, N.dims(), hist_in=2 * FAKE, hist_out=2 * FAKE, vc=2 * FAKE + 32) == 1
    assert _pre(L, N.dims(), kn=3 * FAKE) == 1
    msg = L.gdn_last_error_string().decode()
    assert "overlaps" in msg


def test_scan_rejects_bad_arguments(L):
    from gated_deltanet_linear_pre_gb300 import _native as N
    d = N.dims()
    F = 1 << 26  # buffers 64 MB apart: no accidental overlap
    base = [F, 2 * F, 3 * F, 4 * F, 5 * F, 6 * F]  # qn kn vc glog beta S_in

    def call(S_out=7 * F, o=8 * F, ws=None, ws_bytes=0, T=64):
        return L.gdn_scan(ctypes.byref(d), 1, T, F, *base, S_out, o, ws, ws_bytes, None)

    assert call(o=7 * F) == 1                # o overlaps S_out
    assert "overlaps" in L.gdn_last_error_string().decode()
    assert call(S_out=6 * F + 16) == 1       # partial S_in / S_out overlap
    assert call(o=F) == 1                    # o overlaps qn
    assert call(o=6 * F) == 1                # o overlaps S_in
    need = N.gdn_scan_workspace_bytes(d, 1, 64)
    if need:
        assert call(ws=None, ws_bytes=0) == 4
        assert call(ws=9 * F + 4, ws_bytes=need) == 3


def test_post_rejects_bad_arguments(L):
    from gated_deltanet_linear_pre_gb300 import _native as N
    d = N.dims()
    assert L.gdn_post(ctypes.byref(d), 4, FAKE, 2 * FAKE, 3 * FAKE, 2, 4 * FAKE, None) == 1
    assert L.gdn_post(ctypes.byref(d), 4, FAKE, 2 * FAKE, 3 * FAKE, 0, FAKE, None) == 1
    assert L.gdn_post(ctypes.byref(d), -1, FAKE, 2 * FAKE, 3 * FAKE, 0, 4 * FAKE, None) == 1
    assert L.gdn_post(ctypes.byref(d), 4, FAKE + 4, 2 * FAKE, 3 * FAKE, 0, 4 * FAKE, None) == 3


def test_step_rejects_bad_arguments(L):
    from gated_deltanet_linear_pre_gb300 import _native as N
    d = N.dims()
    F = 1 << 26  # buffers 64 MB apart: no accidental overlap
    # qkv conv_w hist_in hist_out a b z A_log dt_bias gamma S_in S_out y
    good = [F * (i + 1) for i in range(13)]

    def call(n_seq=2, out_f32=0, **kw):
        names = ["qkv", "conv_w", "hist_in", "hist_out", "a", "b", "z", "A_log", "dt_bias", "gamma", "S_in",
                 "S_out", "y"]
        ptrs = [kw.get(nm, good[i]) for i, nm in enumerate(names)]
        return L.gdn_step(ctypes.byref(d), n_seq, *ptrs[:12], out_f32, ptrs[12], None)

    assert call(n_seq=-1) == 1
    assert call(out_f32=2) == 1
    assert call(qkv=None) == 1
    assert call(z=good[6] + 8) == 3
    assert call(hist_out=good[2]) == 1             # history in place is not allowed
    assert "overlaps" in L.gdn_last_error_string().decode()
    assert call(S_out=good[10] + 16) == 1          # partial state overlap
    assert call(y=good[11]) == 1                   # y overlaps S_out
    assert L.gdn_step(None, 2, *good[:12], 0, good[12], None) == 1
    assert call(n_seq=0) == 0                      # empty batch: nothing to do


def test_layer_rejects_small_workspace(L):
    from gated_deltanet_linear_pre_gb300 import _native as N
    d = N.dims()
    need = N.gdn_layer_workspace_bytes(d, 1, 64)
    ptrs = [FAKE * (i + 1) for i in range(13)]
    assert L.gdn_layer(ctypes.byref(d), 1, 64, *ptrs, 0, 20 * FAKE, 30 * FAKE, need - 1, None) == 4


def test_binding_refuses_cpu_tensors():
    import torch
    from gated_deltanet_linear_pre_gb300 import _native as N
    d = N.dims(hk=1, hv=3)
    x = torch.zeros(4, 128, 3)
    with pytest.raises((ValueError, TypeError)):
        N.gdn_post(d, 4, torch.zeros(4, 3, 128), torch.zeros(4, 3, 128, dtype=torch.float16),
                   torch.ones(128), False, torch.zeros(4, 3, 128, dtype=torch.float16))
    del x
