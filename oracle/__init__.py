"""CPU oracle for the quantized paged KV cache -- TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously-correct restatement (numpy; float32 where the
stored codes are decided, float64 for attention) of what the CUDA library
computes, written from the source pages:

  formats    -- INT8 / FP8 E4M3 / FP8 E5M2 per-tensor codes, asymmetric
                INT4 / UINT8 codes with fp16 scale and zero point
  hadamard   -- Sylvester matrix and the fixed-order float32 butterfly
  kvarn      -- variance normalisation + rotation before asymmetric codes
  cache      -- quantize-and-scatter into the paged cache, dequantization
  attention  -- float64 single-token paged decode attention

Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline /
reference leg may import, call or execute anything in this package.  It
shares no code with the CUDA path: the library never imports it, and it
imports nothing from the library.  Pins (tests/test_oracle_*.py) tie every
function to the format definitions, closed forms, library routines and
brute force; there is no function here whose parity is unpinned.
"""
from . import formats, hadamard, kvarn, cache, attention  # noqa: F401
