"""CPU oracle for the 2-bit KV-cache hot path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this package:
only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` may call it.  It shares no code with the CUDA library.

It is a plain, slow restatement of the method, step by step, in numpy:

* ``oracle.kvquant``   rotation, per-channel clip, asymmetric INT2 quantizer
  with fp16 scale/zero, 4-codes-per-byte packing, and the paged tile layout
  the library stores its history in.
* ``oracle.attention`` fp64 softmax attention over the three-tier token pool
  (BF16 sink, INT2 history, BF16 recent) and over an all-BF16 paged cache.
* ``oracle.tiers``     where a newly generated token goes: sink, recent ring,
  or (when the ring is full) eviction of the oldest recent token into history.

Sources: "OSCAR: Offline Spectral Covariance-Aware Rotation for 2-bit KV Cache
Quantization" (gist.science explainer), section 2.2 B "Online-Betriebsphase";
the yunpan.plus practitioner write-up of OSCAR, sections "1. 三段式 Token 池"
and "2. 在线量化与反量化".

Every function is pinned by ``tests/test_oracle_*.py`` to facts that do not
come from the oracle itself (closed forms, brute force, hand-worked fixtures
under ``tests/golden/``).
"""

from . import kvquant, attention, tiers  # noqa: F401
