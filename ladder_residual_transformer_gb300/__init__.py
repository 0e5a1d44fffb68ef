"""GB300-native Ladder Transformer forward pass (prefill and decode).

The compute path is the CUDA library ``libladder.so`` (sm_103a) behind a C ABI
declared in ``include/ladder.h``; ``ladder_residual_transformer_gb300.ladder``
is its thin Python binding; ``checkpoint`` reads Llama-family safetensors
checkpoints into weights for it, and ``timeline`` prints the per-launch decode
timeline.  Submodules load lazily so that importing the synthetic-input
generator does not require a GPU.
"""
__all__ = ["synth", "ladder", "checkpoint", "timeline"]


def __getattr__(name):
    if name in __all__:
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
