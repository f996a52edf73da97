"""CPU oracle for the folded, KV-balanced FP8 MLA decode.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports, links or runs
this package: only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline and reference legs may use it. It shares no code with the CUDA
library or its Python binding; the two meet only through the seeded inputs of
``workloads``.

What it computes, from the pages' problem statement:

* ``e4m3``      -- FP8 E4M3 codes to float64, from the format's bit definition.
* ``attention`` -- exact per-(token, head) softmax attention over the paged
                   latent cache in float64: the absorbed MLA decode is MQA over
                   one 576-dim latent head whose first 512 dims are the value
                   (drafter-attention page, module overview and
                   ``folded_decode``; balanced-MLA page, module overview for
                   the log2 LSE).
* ``merge``     -- the LSE merge of split partials (drafter-attention page,
                   ``DraftDcp``: exp2(lse - max) / sum in FP32 on the pages,
                   float64 here).
* ``uv``        -- the W_UV up-projection of each head's merged latent row
                   (drafter-attention page, ``DraftDcp`` and ``latent_major``).
* ``planner``   -- the integer split planner (balanced and uniform) that the
                   device planner must reproduce bit for bit. The pages name
                   the idea (balanced-MLA page, module overview; rank rule of
                   the drafter-attention page's ``_plan_kernel``) but not the
                   formula; the formula here is this project's reading.

Every function is pinned by ``tests/test_oracle*.py`` to things other than
itself: brute force in pure Python, closed forms, a library routine on a
special case, and invariants (fold = unfold, split-merge invariance,
convexity). No function here is "parity unpinned".
"""
