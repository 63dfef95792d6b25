"""CPU oracle for the routed-MoE forward with per-token NVFP4 activations.

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py`` (its ``cpu_baseline`` leg and
``--impl reference``) may import or run anything in this package.  The CUDA
library (``nvfp4_token_quantized_gb300``) never calls it and has no CPU
fallback; the two share no code.  Inputs for both come from the ``synthetic``
package, which holds random draws only.

* ``oracle.nvfp4`` - E2M1 / E4M3 formats, the per-token / per-expert
  quantizer, bf16 rounding.
* ``oracle.moe`` - router, permutation, expert GEMMs (FP64), SwiGLU,
  requantization, finalize, and the whole forward.

Parity pins (tests that tie the oracle to something other than itself) live
in ``tests/test_oracle_*.py`` and ``tests/golden/``.  Every function here is
pinned; nothing is marked "parity unpinned".
"""

from . import moe, nvfp4  # noqa: F401
