"""Oracle for the quantized MoE layer: plain, slow, FP64 CPU reference.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may use it.  It shares no code with
the CUDA library (no kernels, headers, tables or helpers); it consumes the
same seeded inputs from the ``synth`` module, which holds none of the layer's
arithmetic.

What it computes (DGPP pages, page 1 README "Serves checkpoints as published"
and "Exact"; page 3 README "Execution and performance" table rows
``engine.prefill_bf16_partials`` (per-expert partials summed in fp32 by
default) and ``engine.prefill_fold_scales`` (per-group scale fma by default);
page 4 forum post 1 quantisation table "Activations stay BF16"):

* every weight decoded exactly from its checkpoint format (``formats``);
* router logits as the correctly rounded FP32 value of the exact dot product
  of the BF16 token with the FP32 router row, then softmax, top-k with the
  fixed tie-break (value descending, expert id ascending) and renormalisation
  over the selected experts (``moe.route``);
* the dispatch index as a stable counting sort of (token, slot) pairs by
  expert (``moe.dispatch``);
* per routed pair: gate and up dot products in FP64, SwiGLU in FP64, one
  rounding of the hidden activation to BF16, down projection in FP64, and the
  weighted combine with the FP32 routing weights plus the shared expert,
  rounded once to BF16 (``moe.layer_forward``);
* optionally the fold-scales lever (page 3 README "Execution and performance"
  table, row ``engine.prefill_fold_scales``): int8 g64, FP8 b128 and int4
  g128 weights enter as bf16(fl32(code * scale)) with one accumulator
  (``formats.fold_scales_weights``);
* optionally the NVFP4 W4A4 lever (page 2/3 highlights and page 5 weekly
  update: NVFP4 W4A4 prefill is opt-in): activations and hidden states
  re-quantised to NVFP4 16-element blocks before the projections
  (``moe.nvfp4_quantize_act``).

Parity pins: every function here is checked by ``tests/test_oracle_*.py``
against independent library decoders (torch CPU float8 casts), closed forms,
brute force and exact rational arithmetic.  See the test files for which pin
covers which function.
"""
from . import formats, moe  # noqa: F401
