"""GB300-native (sm_103a) calibration pass for affinity-aware sharding under
Delayed Tensor Parallelism: the head->neuron affinity S_up (FO / ADD) and the
neuron->next-layer-KV-group affinity S_down of one Transformer layer.

The computation lives in libaffinity.so (C ABI, include/affinity.h);
``binding`` is its ctypes binding and ``workloads`` the seeded input
generators.  Importing the package does not load the library.
"""
__all__ = ["binding", "workloads"]
