"""The oracle: a plain, slow, fp64 CPU restatement of the clef-flash prefill forward.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import it.  The CUDA library never calls it and shares no code with it;
the product path fails loudly when its CUDA extension is missing rather than falling back here.

Every step follows the pages' description in the pages' order, written with numpy in float64
(inputs are the exact fp16 values), with no blocking, fusion or reordering beyond the
definitions.  A numpy matmul is used as the library primitive for dense products.

Sources (cited by page title and section in each function):
  * "Clef-Flash-ANE-LUT6" (Hugging Face model card) - Model architecture; Weight precision;
    LUT-6 text weights (the format in ``lut6``, the quantiser in ``quantize``).
  * "clef-flash - Core AI" (README) - Core AI shape (decoder inputs, states, hidden output).
  * "clef-flash-coreml" (README) - decoder parts with cos/sin [L, 64] rotary inputs.
  * "clef-flash-LiteRT" (README) - Host contract (rotary theta 1e7 and the three M-RoPE planes,
    text positions (i, i, i), right padding, the final norm's output per position); Provenance
    (the GatedDeltaNet recurrence in 64-position chunks, grouped keys/values repeated, gated
    full-attention layers).

Functions whose result no page or closed form fixes are marked "parity unpinned" in their
docstring (the end-to-end activations: no page prints any).
"""
from . import lut6, layers, model, quantize  # noqa: F401
