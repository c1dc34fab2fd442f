"""GB300-native MoE-layer forward pass with speculative token shuffling.

The compute lives in ``lib/libsmoe.so`` (hand-written CUDA for sm_103a behind the C
ABI of ``include/smoe.h``); ``binding`` forwards tensors to it. Build it with
``routing_token_shuffle_gb300.build.build()``.

The binding's names are re-exported lazily: importing a submodule that needs no
library (``synth``, ``build``, ``profiling``) neither imports ``binding`` nor maps
``libsmoe.so``; the first use of a binding name does.
"""
import importlib

_BINDING_NAMES = (
    "SMOE_BF16", "SMOE_F32", "LayerIO", "LayerWeights", "SmoeDesc", "SmoeError",
    "desc_from_config", "kernel_launches", "layer_io", "layer_weights", "lib", "make_desc",
    "smoe_combine", "smoe_dispatch", "smoe_ep_exchange", "smoe_expert_ffn",
    "smoe_expert_ffn_gather", "smoe_expert_ffn_gather_fused", "smoe_get_status", "smoe_lar",
    "smoe_layer_forward", "smoe_moe_forward_routed", "smoe_layer_forward_host",
    "smoe_predict_shuffle", "smoe_predict_shuffle_inter", "smoe_predict_shuffle_noalloc",
    "smoe_prefetch_predict", "smoe_route", "smoe_sag", "smoe_selftest_device_timeout",
    "smoe_shuffle_dispatch_rows", "smoe_srs",
    "smoe_token_cluster", "workspace", "workspace_size",
)

__all__ = list(_BINDING_NAMES)


def __getattr__(name):
    if name in _BINDING_NAMES:
        binding = importlib.import_module(".binding", __name__)
        return getattr(binding, name)
    raise AttributeError(f"module {__name__!r} has no attribute {name!r}")
