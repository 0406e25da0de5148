"""Plain CPU oracle of the STILL layer: test infrastructure only.

``ref``   -- the C fp64 streaming recurrence (decode semantics; prefill = N steps).
``brute`` -- NumPy O(N^2) set definition, independent of ``ref``.

Only tests/, the smoke check and the benchmark's CPU-baseline leg import this
package; the CUDA library never does.
"""
