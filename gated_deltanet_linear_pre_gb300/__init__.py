"""GB300-native Gated DeltaNet prompt-prefill path.

The product is the CUDA library libgdn.so (C ABI: include/gdn.h), built for
sm_103a by ``gated_deltanet_linear_pre_gb300.build``.  This package re-exports
its thin ctypes binding under the ABI's names:

    gdn_pre, gdn_scan, gdn_scan_fast, gdn_scan_noalloc, gdn_post, gdn_layer, gdn_layer_fast, gdn_step,
    gdn_scan_workspace_bytes, gdn_layer_workspace_bytes, dims, GdnError

``inputs`` draws the seeded synthetic workloads.  Nothing here computes the
method on the CPU.
"""
_BINDING = ("gdn_pre", "gdn_scan", "gdn_scan_fast", "gdn_layer_fast", "gdn_scan_noalloc", "gdn_post", "gdn_layer", "gdn_step", "gdn_scan_check", "gdn_layer_check", "gdn_scan_noalloc_check", "gdn_last_async_error",
            "gdn_scan_selftest_timeout", "gdn_scan_selftest_one_taker", "gdn_scan_selftest_withhold_flag", "gdn_layer_selftest_stages", "gdn_scan_workspace_bytes",
            "gdn_layer_workspace_bytes", "dims", "gdn_dims", "GdnError", "lib", "library_path")

__all__ = list(_BINDING) + ["inputs", "build"]


def __getattr__(name):
    # the binding (and torch) load on first use, so `inputs` stays light
    if name in _BINDING:
        from . import _native
        return getattr(_native, name)
    raise AttributeError(name)
