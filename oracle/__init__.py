"""Oracle for absorbed MLA decode over a quantized latent KV cache.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check
in ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` may import or run anything in this package.  The CUDA
library never calls it and shares no code with it.

It is a plain, slow, obviously-correct NumPy restatement of what the source
pages (the DeepSeek-V2-Lite "absorbed MLA cache" report in Chinese and English,
and the juejin MLA tutorial) compute:

* ``quant``       - per-(token, group) symmetric INT8, asymmetric INT4 and the
                    comparison quantizers (per-tensor, per-token, symmetric
                    INT4), in IEEE fp32 with round-half-even.
* ``attention``   - weight absorption, absorbed decode (fp64 accumulation),
                    the expanded reference path, split partials and the
                    log-sum-exp combine.
* ``accounting``  - KV bytes per token and capacity arithmetic.

Every function names the passage it follows.  Pins that tie it to something
other than itself live in ``tests/test_oracle_*.py``.  Parity status per
function is listed in each module's header; no function here is "parity
unpinned".
"""

from . import accounting, attention, quant  # noqa: F401
