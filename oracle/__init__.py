"""CPU oracle for the decode-time MoE FFN stage.

TEST INFRASTRUCTURE, not part of the product. It may be imported only by the
tests, by the package's smoke check and by the CPU-baseline leg of the
benchmark; the library never calls it and has no CPU fallback. It is written
from the pages' statement of the method in plain numpy with fp64
accumulation, shares no code with the CUDA sources, and takes its inputs from
the seeded generator.

Pinned functions (tests under tests/test_oracle_*.py pin each one to something
other than itself): rounding helpers, Q4_K / Q5_K / Q8_0 decoding, Q8_1
encoding, integer block dots, router logits, both top-k selections, softmax
over the selected logits, the expert FFN in integer / float / fp16 modes, the
3-input and unfused residual norms, the whole layer with and without a shared
expert (a layer worked out by hand, tests/golden/layer_worked_example.py), and
the parity criteria of parity.py (bf16 spacing from torch's bf16 type, the
boundaries of the float and selection checks). The pages print no worked
example of a whole layer, so the layer's pin is a hand-derived one.
"""
from . import formats, moe  # noqa: F401
