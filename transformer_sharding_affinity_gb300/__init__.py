"""GB300-native (sm_103a) calibration and layout pipeline of affinity-aware
sharding under Delayed Tensor Parallelism: the head->neuron affinity S_up
(FO / ADD / LOO), the neuron->next-layer-KV-group affinity S_down, the layout
objective and search, and the realisation of a layout as sharded weights.

The computation lives in libaffinity.so (C ABI, include/affinity.h).  Modules:
  binding    ctypes binding of every entry point (argument marshalling only)
  scores     one-call s_up / s_down helpers for PyTorch tensors
  stack      a layer stack: calibration with resume, head placement, the
             alternating layout search, realisation of a layer's layout
  shards     merging S computed on disjoint token shards across processes
  workloads  seeded synthetic inputs (no method arithmetic)
  device     host -> device plumbing for those inputs
Importing the package does not load the library.
"""
__all__ = ["binding", "scores", "stack", "shards", "workloads", "device"]
