"""GB300-native Matryoshka contrastive loss (CLIP / SigLIP / row InfoNCE), forward and backward.

The compute lives in a C-ABI CUDA library (``include/uf_contrastive.h``, sources in
``csrc/``); ``binding`` is its thin Python binding and ``synth`` draws seeded inputs.
"""
__version__ = "0.1.0"
