"""CPU oracle for the SpargeAttention2 hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The
product path (the CUDA library and its Python binding) never imports, calls
or links anything here, and nothing here imports the product package.

The oracle is plain NumPy, fp64 by default (fp32 only where a caller asks for
it on large shapes), written from the method's description:

* [P2] "SpargeAttention2: Trainable Sparse Attention via Hybrid Top-k+Top-p
  Masking and Distillation Fine-Tuning" (chatpaper.ai), section "Abstract".
* [P4] "Optimierung der Effizienz von Video-Diffusionsmodellen durch
  SpargeAttention2" (mindverse), sections "Grundlagen der duennbesetzten
  Aufmerksamkeit und ihre Herausforderungen", "Block-duennbesetzte
  Aufmerksamkeit", "Maskierungsstrategien: Top-k und Top-p",
  "Einschraenkungen traditioneller Methoden", "Hybride Top-k+Top-p
  Maskierung", "Effiziente Kernel-Implementierung und Modellanpassung".

Every function is pinned by ``tests/test_oracle_pins.py`` against closed
forms, hand-computed worked examples (``tests/golden/``), brute force on tiny
inputs, library special cases and finite differences.  No function here is
"parity unpinned".
"""

from .sparge_oracle import *  # noqa: F401,F403
from .sparge_oracle import __all__  # noqa: F401
