"""CPU fp64 oracle for one synchronous GPipe training step.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA path; both sides take seeded inputs from ``synth``.

Source of the method: "GPipe technical review" (zzz0906.github.io, a review of
Huang et al., *GPipe: Easy Scaling with Micro-Batch Pipeline Parallelism*).
The review states that synchronous micro-batch accumulation gives exactly the
single-device full-batch result (sections "Preliminaries 6: synchronous vs
asynchronous updates" and "Pipeline flow, phase 3: parameter update"), so the
oracle is that plain definition: one full-batch step, no micro-batches, no
cells, no re-materialisation.

Modules:
  model      full-batch forward / hand-written backward / RMSProp in fp64
  partition  brute-force variance-minimising contiguous partition
  schedule   discrete-event simulation of the pipeline clock (bubble fraction),
             in the GPipe order and the one-forward-one-backward order

Every function here has at least one pin in ``tests/test_oracle_*.py`` that is
independent of the oracle itself (finite differences, an independent autograd
library, closed forms, the review's worked values, brute force).
"""
