"""GDN mixer core for one GB300: conv1d + SiLU, q/k L2 norm, gated delta rule, gated RMSNorm.

The compute lives in libgdn.so (hand-written CUDA for sm_103a, C ABI in
include/gdn.h). ``binding`` marshals torch tensors into it; the ``gdn_*``
names below resolve to the binding on first use, so importing the package
(for example for ``synth``) does not need the built library.
"""
__all__ = ["gdn_conv_update", "gdn_decode_step", "gdn_chunk_prefill", "gdn_spec_verify", "gdn_spec_commit",
           "gdn_gated_rmsnorm", "gdn_state_bytes", "gdn_conv_hist_bytes", "gdn_prefill_workspace_bytes",
           "gdn_read_device_error", "make_dims", "GdnDims", "GdnError"]


def __getattr__(name):
    if name in __all__:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
