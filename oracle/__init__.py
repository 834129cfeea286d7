"""CPU oracle for the rolling FP8 attention cache.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, float64 / explicit
fp32 restatement of what the cache computes, written from the Runway
Characters pages ("Do It Once, at Write Time"; "Where the Time Went";
"Blackwell and Beyond Four GPUs") and the OCP OFP8 format.  Only the tests,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import it.  The CUDA library never imports, links or calls anything here,
and this package imports nothing from the library.

Modules:
  e4m3       FP8 E4M3 encode (RNE, saturating) / decode.
  rope       RoPE table (fp32 from float64 libm) and rotations (pinned fp32,
             exact float64).
  ring       one layer's ring cache: calibrate, write, delta rotate.
  attention  float64 attention over the cache (the reference), the same in
             parts of the slots merged by their log-sum-exps, brute-force
             linear window, the slot-order-positions negative case, and a
             diagnostic that mirrors the kernel's FP8 operand choices.
  legacy     the original upkeep the ring replaced (window copy, RoPE of
             every cached key and re-quantisation at every call).
  projection the QKV projection in front of the cache (bf16 x bf16, summed,
             rounded once to bf16), split into queries, keys and values.

Parity pins: every function here is checked in tests/test_oracle_*.py
against closed forms, invariants, library routines or brute force.  Nothing
in this package is "parity unpinned".
"""
from . import e4m3, rope, ring, attention, legacy, projection  # noqa: F401
from .ring import Ring, INT32_MIN, TO_OLDEST  # noqa: F401
