"""Float64 CPU oracle of one Qwen3-style decoder step.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or
executes this package: it is used by ``tests/``, by ``__graft_entry__.smoke()``
and by the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py``.  It
shares no code, table or helper with the CUDA library; the two meet only at
the seeded input generators of ``decoder_qwen3_step_gb300.inputs``.

Modules
-------
numerics  bf16 / f16 rounding written out from their bit-level definitions
model     the vectorised float64 decoder (numpy), the plain definition
brute     the same decoder in scalar Python loops, for tiny shapes only
compare   the parity metrics (max / mean abs error, argmax with near ties)
int4      int4 group-symmetric weights: quantize, pack, dequantize
sampler   the f64 sampler (penalties, logprob, temperature, top-k, top-p,
          min-p, CDF walk) and its PCG32 streams
"""

from .model import DecoderConfig, Oracle, SeqCache, param_count, rms_norm, rope, attention_one  # noqa: F401
