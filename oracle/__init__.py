"""Float64 CPU oracle for cached incremental causal attention with RoPE.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product path (the CUDA library ``libkvc.so`` and its Python
binding) never imports, links or executes anything here, and nothing here
imports the product package.  The two share no code: the oracle computes its
own RoPE angles, its own rounding to the storage dtype and its own attention.

Sources, cited by page title and section (or listing title) throughout:

* [Ch37] "Keep the prefix, project only the new row" -- learn_llm course,
  chapter 37 (intale.github.io/learn_llm/en/course/37-incremental-attention/;
  the Russian page of the same chapter prints byte-identical listings).
* [LCP5] "LLM 机制实验（五）：改了历史，能否只重算变化的后缀？"
  (huhohoo.com/docs/llm/longest-prefix-reuse).

What each module computes and what pins it (tests/test_oracle_*.py):

* ``rope``      RoPE at absolute positions.  Pinned: the rotation direction and
                offset by the [Ch37] fixture trace, the 2-D case by the closed
                form, the block structure by a matrix exponential.
* ``storage``   rounding to the cache storage dtype (bf16 / f32 / f64).
                Pinned against torch's float32->bfloat16 cast and brute force.
* ``attention`` newest-query attention, full masked causal attention, the
                decode and suffix-chunk definitions, GQA head map.  Pinned by
                the [Ch37] printed weights/outputs, torch's SDPA (fp64) and
                closed-form special cases.
* ``prefix``    longest-common-prefix cut, truncation, projection counts.
                Pinned by the [LCP5] table and brute force.
* ``toy_decoder`` the 2-layer single-head decoder of [LCP5].  Pinned by
                cached == recomputed (<= 1e-12), causality and the table's cuts
                and counts.  The two negative-control magnitudes the page
                prints (1.37749785, 0.64189345) depend on weights the page does
                not publish: parity unpinned for those two numbers; only
                "error > 1e-12" is checked.
* ``fixture``   the [Ch37] 1-layer, 2-head, d_h = 2 fixture replay.
"""

from . import rope, storage, attention, prefix, toy_decoder, fixture  # noqa: F401
