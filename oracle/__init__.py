"""CPU oracle for exact attention (forward and backward) -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the C-ABI library and
its Python binding) never calls it, and it shares no code with the CUDA path:
it takes plain numpy arrays and returns plain numpy arrays.

Contents (all arithmetic in float64 unless a format fixes otherwise):
  attention  -- three-pass safe-softmax attention, the plain definition
                (scores, row max, sum of exponentials, weighted sum of values,
                logsumexp); plus the streaming (m, l, o) recurrence and the
                blockwise merge rule, used only to pin the three-pass routine.
  hadamard   -- Sylvester Hadamard matrix and the fast Walsh-Hadamard transform.
  e4m3       -- exact FP8 E4M3 encode (round-to-nearest-even, saturating) and
                decode.
  fp8        -- incoherent processing (random-sign Hadamard rotation) and
                per-128-row-block E4M3 quantisation of Q, K, V; dequantisation.
  backward   -- gradients dQ, dK, dV of attention given dO: the chain rule
                through the row softmax written out (the backward pass).

Pins: every function here is checked by the ``-m "not gpu"`` tests against
facts the source pages or mathematics fix (a printed worked example, closed
forms, invariants, library routines).  No function is "parity unpinned".
"""
from . import attention, backward, e4m3, fp8, hadamard  # noqa: F401
