"""GB300 (sm_103a) kernels of the weight-bound verify forward of greedy
speculative decoding, behind the C ABI of ``include/sdv.h`` (``libsdv.so``).

``sdv`` is the Python binding (argument marshalling only); ``build`` compiles
the library in-tree with nvcc.
"""
from . import sdv  # noqa: F401
from .sdv import QWeight, SdvError  # noqa: F401
