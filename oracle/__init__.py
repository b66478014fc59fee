"""Oracle: a plain CPU restatement of TurboQuant-style KV-cache compression
and compressed-KV decode attention.

TEST INFRASTRUCTURE.  Nothing on the product path may import, call or run
anything in this package: only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py`` (its ``cpu_baseline`` leg and its ``--impl reference`` arm) use
it.  It shares no code, tables or constants with the CUDA library; the two
meet only through the seeded inputs of the ``synth`` package and through
bytes in the documented page layouts.

Arithmetic is numpy float64 unless a stored format fixes the precision: the
value group quantiser and the affine int8 key quantiser run in IEEE float32
(both sides make those integer decisions in the same precision), norms and
scales are rounded to fp16 where the layout stores fp16.

Modules and the passages they follow (page titles as printed on the pages):

* ``rotation``  random-sign diagonal + normalised Walsh-Hadamard transform
  ("TurboQuant-MLX overview", PolarQuant step 1; turboquant vLLM guide, §二
  step 1).
* ``codebook``  Lloyd-Max codebook for the coordinate density of a rotated
  unit vector (turboquant vLLM guide, §二 step 2, "Beta-distribution optimal
  codebook").
* ``rng``       SplitMix64 counter generator for the random signs and the
  Gaussian sketch matrix (the pages do not fix a generator).
* ``quant``     key encoder (Lloyd-Max + QJL residual sign sketch), value
  group quantiser, alternate-layout encoders (vllm-metal TurboQuant guide,
  quantisation principle table).
* ``layout``    generic low-bit packing and the page-tile byte layouts.
* ``attention`` decode attention over the compressed cache plus the exact
  recent-token buffer.

Pins (``tests/test_oracle_*.py``): each function is checked against something
other than itself -- closed forms, textbook tables, library routines, brute
force, the pages' printed byte counts.  Functions without such a pin are
marked "parity unpinned" in their docstring; currently none is.
"""
from . import attention, cache, codebook, layout, quant, rng, rotation  # noqa: F401
