"""CPU oracle for the DeepSeek V4.1 Engram forward path.

THIS IS TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT. Only the tests, ``__graft_entry__.smoke()``
and the benchmark's CPU-baseline leg may import it. It shares no code with the CUDA path
(``deepseek_v4_engram_gb300``) and neither imports the other.

It is a plain, slow restatement of what the Engram pages define, in float64 numpy, one function
per stage, each citing the passage it follows:

* :mod:`oracle.numerics` - bf16, fp8 e4m3fn and e8m0 encodings from their bit fields.
* :mod:`oracle.engram`   - the n-gram hash with its look-back cache, the table-row gather and
  dequantisation, the bf16 ``wkv`` projection, and the gate-and-add.

Every function is pinned by ``tests/test_oracle_*.py`` to facts the pages and the mathematics fix
(closed forms, library casts on the cases where they coincide with the definition, invariants),
not to a retyping of itself. One part is "parity unpinned": no real hash tables or golden
captures exist here, so the hash is pinned to its stated structure only, never to the model's
actual tables.
"""
from . import engram, numerics  # noqa: F401
from .engram import NgramHashState, embed_rows, forward, gate_and_add, linear_bf16  # noqa: F401
