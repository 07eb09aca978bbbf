"""Plain fp64 CPU oracle for the ReLU activation-sparse feedforward layer.

TEST INFRASTRUCTURE ONLY. Nothing in the library imports, calls or links this
package; only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may use it. It shares no code with the
CUDA path: the only module both sides use is the seeded input generator in
``synthetic/``, which holds none of the FFN arithmetic.

Modules
-------
``ffn``      dense definition of the forward pass (gated and non-gated) and of the
             gradient of  L = sum(dy * y) + l1 * sum(a),  in float64.
``formats``  TwELL (tile-wise ELLPACK) and Hybrid (compact ELL + dense backup)
             packing and unpacking, as the pages define the formats.
``sparse``   the same forward/backward computed entry by entry from the packed
             formats (the method is exact: it only skips multiplications by zero).
``neurons``  per-neuron activity counts and the dead-neuron re-initialisation of
             the gate projection (a counter-based SplitMix64 / Irwin-Hall draw).

Every function here is pinned by ``-m "not gpu"`` tests against something other
than itself (brute force, closed forms, finite differences, a hand-worked fixture,
invariants, torch autograd); see the test files ``tests/test_oracle_*.py``.
"""
from . import ffn, formats, neurons, sparse  # noqa: F401
