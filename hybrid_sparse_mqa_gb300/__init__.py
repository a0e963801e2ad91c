"""GB300-native hybrid sparse MQA attention step (DeepSeek-V4 decode / verify).

The compute path is the C-ABI library ``libdsv4attn.so`` built from ``csrc/``;
``hybrid_sparse_mqa_gb300.attn`` is its Python binding.  ``synth`` draws seeded
synthetic inputs.  Importing the package does not load the library.
"""
__all__ = ["attn", "synth"]
