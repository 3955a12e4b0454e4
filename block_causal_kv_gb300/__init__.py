"""GB300-native hot path of D2F block-diffusion decoding.

Block-causal attention over a paged KV cache, the confidence commit over the
vocabulary, and the append of finished blocks, as hand-written sm_103a CUDA
kernels behind a C ABI (libd2f.so). This package is the thin Python binding
(argument marshalling only) plus seeded synthetic inputs.

  from block_causal_kv_gb300 import d2f   # the binding; loads libd2f.so
  from block_causal_kv_gb300 import synth # seeded workloads
"""
import importlib

__all__ = ["d2f", "synth"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module("." + name, __name__)
    raise AttributeError(name)
