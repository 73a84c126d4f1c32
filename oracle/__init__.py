"""Float64 CPU oracle of the Mamba-2 SSD core (forward + analytic backward).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg may import this package; the CUDA library never does, and
the two share no code.

* ``oracle.ssd_oracle.c`` — the sequential recurrence and its reverse-time
  adjoint in plain C (float64), built on demand with gcc.
* ``oracle.core`` — ctypes wrapper taking numpy float64 arrays.
* ``oracle.dual`` — an independent numpy restatement of the forward as the
  quadratic ("dual") form, for brute-force checks on tiny inputs.
"""
from .core import build_oracle, ssd_forward, ssd_backward, default_threads  # noqa: F401
