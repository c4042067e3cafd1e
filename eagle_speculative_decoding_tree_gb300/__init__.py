"""EAGLE draft-tree verify step on one GB300 (sm_103a).

The compute lives in libeagle.so (CUDA kernels behind the C ABI of include/eagle.h);
``binding`` is the thin Python layer with the ABI's names, ``step`` strings the
calls of one verify step together, and ``synth`` draws seeded synthetic inputs.
"""
__all__ = ["binding", "build", "step", "synth"]
