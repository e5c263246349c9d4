"""CPU oracle for the batched W4A16 MoE decode step.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may use it.  It shares no code with the CUDA library.

What it is: a plain, slow, fp64 numpy restatement of what the decode step
computes, written from these pages (cited by abbreviated title):

* [KV-slot isolation] "Per-stream KV-slot isolation for parallel low-bit
  decode on Apple Silicon: crash fix with byte-identical solo parity and
  no-regression"
* [Crash root cause] "A falsify-first root cause for a concurrent 4-bit decode
  crash: batch-composition KV-pool wipe trips a re-seed precondition"
* [Batched serving] "Batched-concurrent 4-bit serving on Apple Silicon:
  weight-stream amortization with an honest sublinear ceiling"

The pages' Methods sections are empty, so the arithmetic of each step is the
plain reading of the op each page names (packed-int4 weights with per-group
scales, a batched dense GEMM, top-k expert routing, a grouped expert op, slot
attention, a per-stream output projection, greedy decode).  Every reading
taken where the pages are silent is listed in the module that takes it.

Pinning: every function here is checked by ``tests/test_oracle_*.py`` against
hand-computed fixtures (``tests/golden/``), closed forms, invariants and brute
force on tiny inputs.  One function is "parity unpinned": the end-to-end model
output against a real checkpoint (no trained weights exist here).
"""

from .numerics import (bf16_round, bf16_bits, from_bf16_bits, unpack_int4,
                       pack_int4, dequant_w4, quantize_w4)
from .ops import (w4_gemm, rmsnorm, rope_rotate_half, slot_attention, causal_block_attention,
                  silu, route_topk, expert_ffn, moe_combine)
from .model import (OracleConfig, OracleSlotMap, OracleKV, decoder_layer, moe_block, lm_head_logits,
                    model_step, prefill_layer, model_prefill)

__all__ = [
    "bf16_round", "bf16_bits", "from_bf16_bits", "unpack_int4", "pack_int4",
    "dequant_w4", "quantize_w4", "w4_gemm", "rmsnorm", "rope_rotate_half",
    "slot_attention", "causal_block_attention", "silu", "route_topk", "expert_ffn", "moe_combine",
    "OracleConfig", "OracleSlotMap", "OracleKV", "decoder_layer", "moe_block", "lm_head_logits", "model_step",
    "prefill_layer", "model_prefill",
]
