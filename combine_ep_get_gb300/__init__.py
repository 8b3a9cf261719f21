"""GB300-native MoE token dispatch / combine (layout -> dispatch -> combine).

The compute path is the CUDA library ``libep_get.so`` (sm_103a kernels behind
a C ABI declared in ``include/ep_get.h``).  ``combine_ep_get_gb300.binding``
is a thin ctypes layer over it with the same entry-point names; importing it
fails loudly when the library has not been built.  There is no CPU fallback.

``combine_ep_get_gb300.inputs`` draws seeded synthetic inputs and does not
load the library.
"""

_BINDING_NAMES = (
    "ep_get_layout", "ep_dispatch", "ep_combine", "ep_layout_and_dispatch", "ep_layout_workspace_bytes",
    "ep_recv_capacity_bound", "ep_status_string", "Layout", "alloc_layout",
    "ep_get_layout_static_scratch", "ep_dispatch_expanded", "ep_combine_expanded",
    "ep_expanded_capacity_bound", "ep_combine_topk_weights", "ep_accumulate_expert_stats",
    "ep_bounds_checked", "EP_BF16", "EP_FP8_E4M3",
)


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
