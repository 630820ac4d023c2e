"""GB300 (sm_103a) library for the hybrid-tree speculative-decoding verify step.

The compute path is libgraft.so (hand-written CUDA, C ABI in include/graft.h);
``binding`` wraps its entry points one-to-one, ``step.VerifyStep`` chains
them into one step, ``synth`` draws the seeded synthetic inputs and
``_build`` compiles the library in-tree with nvcc.
"""
__all__ = ["binding", "step", "synth"]
