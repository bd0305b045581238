"""Plain fp64 CPU oracle for the OSCAR INT2 rotated KV-cache hot path.

TEST INFRASTRUCTURE ONLY.  This package is the slow, obviously-correct
restatement of what the hot path computes.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py`` (its CPU-baseline leg and its
``--impl reference`` arm) may import it.  The product package
``int2_rotated_kv_oscar_gb300`` never imports it, and nothing here imports
the product: the two share no code, headers, tables or constants.  The only
thing both sides consume is data made by the seeded input generators.

Sources (the pages the method is defined on; cited by title and section):

* [IT]  ainsights.it, "OSCAR: Come Together AI Comprime la KV Cache a 2-bit
  per LLM" -- sections "I tre fattori della rotazione" (the three factors),
  "Architettura del Sistema di Serving e Layout di Memoria" (sink / recent /
  history layout, fused write and read kernels), "Guida Rapida" (server flags
  ``--oscar-sink-size 64``, ``--oscar-recent-size 256``).
* [RU]  edge.aivizor.me, "Together AI выпустила исходники OSCAR — INT2-квантование
  KV-кэша для долгих контекстов LLM" -- paragraph "Техническая идея" (C_Q, C_S,
  eigenbases), the composition paragraph (R_K = U_Q H P, R_V = U_S H P), the
  deployment paragraph (lemma diag = tr(Lambda)/d, sink S0 = 64).
* [ES]  gist.science, "Resumen Técnico: OSCAR - Rotación Consciente de la
  Covarianza Espectral Offline para Cuantización de Cache KV de 2 bits" --
  §2.1 (Q^T Q and V^T S^T S V objectives), §2.2 A (offline calibration steps
  1-4), §2.2 B (mixed-precision paged cache, fused kernel).

Modules:

* ``rotation``    Walsh-Hadamard, bit reversal, R = U H P, x' = x R.
* ``quant``       per-group clip + fp16 scale + 4-level code; dequantisation.
* ``layout``      the paged INT2 block byte layout (written from the layout
                  specification in the C header's documentation, as a
                  (token, channel) -> (byte, bit) map).
* ``cache``       sink / recent / history segments; the append/eviction model.
* ``attention``   softmax attention in fp64; decode over a mixed cache.
* ``calibration`` offline C_Q, C_S, eigenbases and clip thresholds.

Every public function is pinned by a ``-m "not gpu"`` test in
``tests/test_oracle_*.py`` against something other than itself (closed
forms, textbook special cases, brute force, hand-worked golden fixtures).
Functions without such a pin say "parity unpinned" in their docstring; at
present there are none.
"""

from . import rotation, quant, layout, cache, attention, calibration  # noqa: F401
