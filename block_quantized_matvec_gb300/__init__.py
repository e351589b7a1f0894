"""GB300-native block-quantized matrix-vector products (MMVQ) at 1-8 columns.

The compute path is the C-ABI library ``libmmvq.so`` (CUDA, sm_103a) built
from ``csrc/``; :mod:`.mmvq` is its thin Python binding.  Importing this
package does not load the library: the first call into :mod:`.mmvq` does,
and raises if it is missing.  There is no CPU fallback.
"""
