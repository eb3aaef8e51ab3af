"""CPU oracle for the low-bit weight GEMV/GEMM path -- TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct restatement of what the path computes, in fp64, written
from the pages and independent of the CUDA path (no shared code, headers, tables or
constants; neither side imports the other).  Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import it.  The product path never calls it.

Modules
  numerics  -- fp16/bf16 decoding and round-to-nearest-even into bf16.
  int4      -- symmetric per-group INT4: dequantise, multiply, pack/unpack the layout.
  binplane  -- ShiftAdd binary planes: dequantise, multiply, pack/unpack the layout.
  sa        -- the deployed ShiftAdd format (u8 scale codes x one fp16 d per 256 inputs):
               dequantise, multiply, pack/unpack the layout.
  nvfp4     -- NVFP4 weights (E2M1 x E4M3 per 16 x fp32) and the trimmed draft head's
               argmax through an id map: dequantise, multiply, pack/unpack the layout.
  q8        -- Q8 weights for the draft head (int8 x one fp16 scale per 32 inputs):
               dequantise, multiply, pack/unpack the layout.
  verify    -- vocabulary argmax (lowest index on ties), greedy prefix acceptance, and the
               merge of a row-sharded head's slice winners.

Parity pins (tests/test_oracle_pins.py) tie every function to something other than
itself: hand-worked 4x8 examples, brute force on tiny shapes, closed forms, invariants
and library rounding routines.  No function here is "parity unpinned".
"""
from . import numerics, int4, binplane, sa, nvfp4, q8, verify  # noqa: F401
