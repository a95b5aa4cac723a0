"""CPU oracle for the exact attention forward — TEST INFRASTRUCTURE ONLY.

This package is the slow, obviously-correct statement of what the GPU path
computes.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import or run it; the product path (the C-ABI library
and its Python binding) never does, and it shares no code with it.

Modules
-------
attention  the plain definition in float64 (materialised scores, two-pass
           row softmax), plus row-sampled and probability-matrix variants.
online     the tile-by-tile online-softmax recurrences printed on the pages,
           in float64, used only to pin the definition against the method.
brute      a pure-Python triple loop (``math.exp``), for tiny shapes.

Sources (titles of the pages this follows):
  * "flash attention v3 paper" search page (cidian.kuaisou.com), first
    snippet: the standard attention definition S = QK^T, P = rowsoftmax(S),
    O = PV, with scale and mask omitted before the softmax.
  * "Flash Attention (Kutarisa Kwemheni)" explainer (aiunderstanding.org),
    summary and FAQ: the method is exact attention computed with tiling and
    an online softmax.
  * "Hacker News Digest — gpu-computing" (hckr.top), section "Алгоритм Flash
    Attention 2" (pseudocode: scale = DIM**-0.5 applied to Q K^T) and section
    "v1 — базовая версия", item 3 (the running max / denominator recurrence).

Parity status: every public function here is pinned by CPU tests against
closed forms, invariants, a library routine and the brute force; none is
"parity unpinned".  ``probabilities_fp64`` is pinned by hand-derived weight
matrices (tests/golden/closed_forms.json, field "p", including a
grouped-query case whose kv heads differ) and by P V equalling the output of
plain multi-head attention on repeated K/V; planted mistakes in its scale,
head map, normalisation axis and mask fail those pins.
"""

from .attention import (  # noqa: F401
    attention_fp64,
    attention_rows_fp64,
    probabilities_fp64,
    kv_head_index,
    visible,
)
from .online import online_normalised_fp64, online_deferred_fp64  # noqa: F401
from .brute import attention_loops  # noqa: F401
