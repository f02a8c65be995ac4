"""relation-aware self-attention on GB300 (sm_103a): the Shaw forward, T5 / ALiBi /
per-offset scalar biases, labelled edges, a decode step, the Shaw gradients and those
of labelled edges and the scalar biases.

The compute lives in librelattn.so (C ABI, include/relattn.h); this package holds its
ctypes binding (`_lib`), the in-tree build script (`build`) and the named workloads with
their seeded input generator (`workloads`). The binding is imported lazily so that
`workloads` can be used without the compiled library; touching a binding function when
the library is not built raises ImportError.
"""
from __future__ import annotations

_BINDING = ("relattn_fwd", "relattn_t5bias_fwd", "relattn_alibi_fwd",
            "relattn_offset_bias_fwd", "relattn_labeled_fwd", "relattn_txl_fwd", "relattn_sinusoid_table",
            "relattn_decode_fwd",
            "relattn_decode_fwd_noalloc", "relattn_decode_workspace_size", "relattn_bwd",
            "relattn_bwd_workspace_size", "relattn_scalar_bias_bwd",
            "relattn_scalar_bias_bwd_workspace_size", "relattn_labeled_bwd",
            "relattn_labeled_bwd_workspace_size", "relattn_labels",
            "relattn_t5_thresholds", "relattn_set_wait_limit",
            "relattn_debug_withhold_first_load", "relattn_set_short_kernel",
            "relattn_set_bwd_tensor_cores",
            "relattn_get_device_error", "relattn_status_string", "relattn_version",
            "RelattnError")

__all__ = list(_BINDING)


def __getattr__(name):
    if name in _BINDING:
        from . import _lib
        return getattr(_lib, name)
    raise AttributeError(name)
