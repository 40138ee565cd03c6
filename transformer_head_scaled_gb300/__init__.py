"""GB300-native (sm_103a) multi-head scaled dot-product attention forward.

The compute path is the CUDA library built from ``csrc/`` (a C ABI declared in
``include/attn.h``); this package only builds it and marshals arguments to it
through ctypes.  Importing the package does not load the library: the first
call to :func:`attn_fwd` (or :func:`load`) does, and raises if it is missing.
"""
from .inputs import MASK_CAUSAL, MASK_KEY_PADDING, MASK_NONE  # noqa: F401


def __getattr__(name):
    if name in ("attn_fwd", "attn_fwd_f32", "attn_fwd_raw", "attn_fwd_f32_raw", "attn_decode",
                "decode_workspace_bytes",
                "load", "AttnError", "status_string", "check"):
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
