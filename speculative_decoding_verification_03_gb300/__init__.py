"""GB300-native batched speculative-decoding verification with the fused
Adaptive-Verification acceptance estimator.

The compute path is the C-ABI library ``libspecverify.so`` (hand-written CUDA
for sm_103a); :mod:`.binding` marshals torch tensors into it.  Importing the
package does not load the library; the first call into :mod:`.binding` does,
and raises if the library was not built.
"""
__all__ = ["binding", "synth"]
