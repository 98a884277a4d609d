"""CPU oracle of the TriAttention KV-cache eviction pass.

TEST INFRASTRUCTURE, NOT PRODUCT CODE. Only ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline / reference leg may import it. The product path
(the CUDA library and its Python binding) never imports, links or calls it, and
this package never imports the product.

It is plain, slow and obviously correct: numpy in float64, the method's steps
in the order the pages give them, library primitives (matmul, stable sort)
used only as whole steps. See :mod:`oracle.tria_oracle`.

Pin status: every function is pinned by a test against a brute-force or
closed-form computation, an identity the pages rely on, or a value the pages
print - the pass in ``tests/test_oracle_pins.py``, the decode-loop schedule in
``tests/test_lifecycle.py``, the shared-slot combine in
``tests/test_shared_oracle.py`` (by its reduction to the per-segment pass and
the max identity; the combine rule itself is a reading, the pages state none)
- except the reading of the future-offset set D (the pages do not state D; it
is a load-time parameter and both sides take the same D), which is a
documented reading rather than a pinned value.
"""
from .tria_oracle import *  # noqa: F401,F403
