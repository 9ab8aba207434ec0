"""CPU oracle for trie-constrained greedy decoding (test infrastructure only).

This package is a plain, slow, obviously-correct restatement of what the
constrained decode step computes.  It exists to check the CUDA path and is not
part of the product: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference arm of ``bench.py`` may import it.  It shares no code
with the CUDA path (no kernels, headers, tables or helpers); the two meet only
in the seeded input generators, which hold none of the method's arithmetic.

Modules:

* ``oracle.language`` - the finite language of k-pointer outputs and the
  next-token mask taken literally from its definition (brute force).
* ``oracle.grammar``  - the catalog as a prefix trie (dicts of sets), the
  compile-time refusals, and the per-step legal set and transition of the
  tool-pointer walk.
* ``oracle.head``     - bf16 decoding, exact fp64 logits of candidate rows, the
  lower-id tie-break argmax, and the dense-logits-then-mask baseline.
* ``oracle.decode``   - the greedy decode loop, the host replay check and the
  teacher-forcing comparison used for floating-point parity.
* ``oracle.sample``   - sampling with temperature, top-k and top-p and their
  tie rules, the sampling decode loop and its teacher-forcing checker.
* ``oracle.chars``    - the character-level constraint over a byte vocabulary
  (every tokenization of a catalog string accepted), from its definition, and
  brute-force enumeration of its language.

Every function is pinned by a ``-m "not gpu"`` test against something other
than itself (brute-force enumeration, exact integer arithmetic, constructed
ties, hand-derived fixtures under ``tests/golden/``).
"""

from . import language, grammar, head, decode, sample, chars  # noqa: F401
