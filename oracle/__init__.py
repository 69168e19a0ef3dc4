"""CPU oracle for the speculative-decoding verify path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product (the C-ABI library, its
Python binding) imports, calls or links anything in this package; only the
tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
use it.  It shares no code with the CUDA path: the two meet only in the
seeded input bytes that ``synth`` generates.

It is a plain, slow restatement of what the pages define, in float64 where
the pages leave the precision open, written in plain C++
(``oracle/src/oracle.cpp``, built by ``oracle/build.py`` into
``liboracle.so``): fp64 sums term by term in reduction order, no BLAS, no
blocking, no vector intrinsics; OpenMP spreads output rows over threads and
leaves every element's arithmetic unchanged.  The Python modules below only
marshal numpy arrays into it (``_native``):

* ``quant``   -- per-block-32 absmax symmetric int8 / int4 quantisation and
                 the int4 nibble packing;
* ``verify``  -- the dequantised skinny GEMM over the S = K+1 verify window,
                 the per-row argmax and the greedy longest-prefix accept;
* ``mlp``     -- SiLU, the SwiGLU gate/up projection and the top-k routed
                 gathered-expert MoE;
* ``sample``  -- the sampling (temperature > 0) verify and its counter-based
                 random numbers;
* ``spec_loop`` -- a toy greedy speculative-decoding loop (n-gram drafter,
                 fused a0 scheme) used to pin the accept step against plain
                 greedy decoding (Python test machinery around the C++ argmax
                 and accept).

Every function's docstring names the page and section it follows and the
reading taken where the pages are silent.
"""

from . import quant, verify, mlp, sample, spec_loop  # noqa: F401
from ._native import set_threads, threads  # noqa: F401
