"""CPU oracle for the hybrid-tree verify step (test infrastructure only).

This package is the plain, slow, obviously correct definition of what the
GPU library computes.  It exists so that tests, the smoke check and the CPU
baseline of the benchmark have something independent to compare against.
Nothing in the product path may import it: only ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference leg of
``bench.py`` use it.

It shares no code with the CUDA library and imports nothing from the
``tree_verification_gb300`` package; inputs are handed in as NumPy arrays.

Sources.  The method is described by two web pages on one paper:

* "Draft Less, Retrieve More: Speculative Decoding을 위한 하이브리드 트리 구성"
  (aitrends.kr article; cited below as *Graft article* with its paragraph:
  lead, step summary, method, results, architecture);
* "Draft Less, Retrieve More: Hybrid Tree Construction for Speculative
  Decoding" (chatpaper.ai abstract; cited as *Graft abstract*).

The pages fix the shape of the method but not its formulas.  Every point
they leave open is resolved by a stated reading in the docstring of the
function that needs it.

Modules:

* ``config``     budget split Kmax = K_draft_s + K_ret_s and retrieval templates
* ``tree``       draft-tree build with dynamic-depth pruning, retrieval, merge
* ``attention``  tree-masked GQA attention (softmax definition, fp64)
* ``accept``     greedy longest-accepted-path and KV compaction
* ``update_m``   online update of the adjacency table M
* ``step``       one whole verify step composed from the above
* ``tiny_lm``    a tiny random-init transformer used for the losslessness pin

Parity status: every function here is pinned by a test in
``tests/test_oracle_*.py`` against something other than itself (brute force,
a library routine, a closed form or a hand-worked fixture).
"""
