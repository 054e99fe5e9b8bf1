"""GB300-native routed mixture-of-experts FFN over a prompt chunk.

The compute runs in the CUDA library ``libmoe_gb300.so`` (see
``routed_expert_prefill_gb300.moe`` for the Python binding).  Importing this
package does not load the library; ``import routed_expert_prefill_gb300.moe``
(or touching one of the names below) does.
"""

__all__ = ["moe_route_topk", "moe_build_csr", "moe_experts_fwd"]


def __getattr__(name):
    if name in __all__:
        from . import moe

        return getattr(moe, name)
    raise AttributeError(name)
