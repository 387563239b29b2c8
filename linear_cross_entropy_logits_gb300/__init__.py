"""GB300-native fused linear cross entropy (FLCE): forward and backward of a language-model
head without materialising the [BT, V] logits.

The compute path is the C-ABI library ``libflce.so`` (hand-written sm_103a CUDA); this
package holds its thin ctypes binding (``flce``), the build step (``build``) and the seeded
input generators (``inputs``). Importing the package does not load the library; the first
call into ``flce`` does, and fails loudly if it has not been built.
"""

__all__ = ["flce", "inputs", "build"]
