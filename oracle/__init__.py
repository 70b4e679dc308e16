"""The oracle: a plain, slow, fp64 CPU restatement of the clef-flash prefill forward.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
legs of ``bench.py`` may import it.  The CUDA library never calls it and shares no code with it;
the product path fails loudly when its CUDA extension is missing rather than falling back here.

The oracle is plain C++17 with OpenMP (``oracle/csrc``, built into ``oracle/liboracle.so`` by
``oracle/build.py``), every product and sum in float64, the inputs the exact fp16 values.  Every
step follows the pages' description in the pages' order with no blocking, fusion or reordering
beyond the definitions: the gated delta rule as the per-token recurrence, attention as one
explicit softmax per query row, each GEMM output one dot product.  The Python modules
``lut6``, ``layers``, ``model``, ``quantize`` and ``head`` only marshal numpy arrays into its C ABI
(``oracle/csrc/oracle.h``).

``oracle/twin`` is a second, independent writing of the same definitions in numpy; it is used
only by ``tests/test_oracle_twin.py`` to cross-check the C++ oracle.

Sources (cited by page title and section in each function):
  * "Clef-Flash-ANE-LUT6" (Hugging Face model card) - Model architecture; Weight precision;
    LUT-6 text weights (the format, and the quantiser).
  * "clef-flash - Core AI" (README) - Core AI shape (decoder inputs, states, hidden output).
  * "clef-flash-coreml" (README) - decoder parts with cos/sin [L, 64] rotary inputs.
  * "clef-flash-LiteRT" (README) - Host contract (rotary theta 1e7 and the three M-RoPE planes,
    text positions (i, i, i), right padding, the final norm's output per position); Provenance
    (the GatedDeltaNet recurrence, grouped keys/values repeated, gated full-attention layers).

Functions whose result no page or closed form fixes are marked "parity unpinned" (the
end-to-end activations: no page prints any).
"""
from . import head, layers, lut6, model, quantize  # noqa: F401
