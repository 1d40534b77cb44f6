"""CPU oracle for exact attention (float64).  TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library and its Python binding
never import it, and it imports nothing from them.

* ``oracle.attention`` - the plain three-step definition (scores, softmax,
  weighted values) with the natural-log LSE; this is what every GPU result is
  compared with; ``attention_fwd_gqa`` is the same per query head with K/V
  heads shared by groups of query heads.
* ``oracle.online`` - the online-softmax recurrence and the split combine,
  used only by tests to pin that streaming equals the plain definition.

Every function here is pinned by ``tests/test_oracle_*.py`` to values the
pages print, to closed forms, to invariants and to brute force on tiny inputs.
"""
from .attention import attention_fwd, attention_fwd_gqa, attention_head, probabilities  # noqa: F401
