"""Oracle: a plain, slow CPU restatement of the block-quantized decode step.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import or run this package.  The product
path (the CUDA library and its Python binding) never imports it, never calls
it, and shares no code, table or helper with it; the only thing both sides use
is the seeded input generator in ``synth``.

What it computes, and where that is defined:

* ``quant``   -- the Q8_0 / Q4_0 block formats (GGUF-style blocks of 32 along
  the input dimension, one fp16 scale per block), as the workload
  descriptions define them; encoding and decoding.
* ``model``   -- the Qwen3-style decoder forward pass, step for step as the
  pages print it: embedding lookup, pre-norm blocks with RMSNorm, Q/K/V
  projections, per-head QK-RMSNorm before half-split RoPE, KV cache append,
  grouped-query attention with a causal mask in prefill, output projection
  and residual, SwiGLU FFN and residual, final RMSNorm, tied LM head, greedy
  argmax ("Всередині LLM: чисте виконання на Python для Qwen3-0.6B на MLX",
  steps 2-9; "Inferencia local y arquitecturas", section "El formato",
  qwen3.archdef).  Weights are dequantized and multiplied in floating point
  with no activation quantization ("Inferencia local y arquitecturas",
  section "Elegir el motor").

Default precision is float64.  Pins: ``tests/test_oracle_*.py``.
"""
from . import quant, model  # noqa: F401
from .quant import (quantize_q8_0, quantize_q4_0, dequantize, quantize)  # noqa: F401
from .model import OracleModel, run_greedy  # noqa: F401
