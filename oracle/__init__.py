"""CPU oracle for decode_step_batch — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg (and its ``--impl reference`` arm) may import anything from here. The
product library neither imports nor links this package, and this package
imports nothing from the product library.

Contents:
  oracle.cpp   plain C++17 f32 model (serial Step, panel StepBatch, sampler,
               Q8_0 quantiser, Philox4x32-10), built with -ffp-contract=off
  core.py      ctypes binding of oracle.cpp
  pages.py     page-allocator model (lowest free index first)
  sched.py     scheduler references: fill / gather / fold over the oracle
               model, and the model-free tick simulation
"""
