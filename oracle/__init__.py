"""CPU oracle for the sparse-attention decode path (TEST INFRASTRUCTURE ONLY).

Plain, slow, sequential numpy/Python code in float64 that states what each step
of the path computes. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import it; the product package never does, and
this package shares no code with the CUDA path (the seeded input generators in
``synth`` are the only thing both sides use).

Sources (page titles; section headings given in the original and in English):

* [P3] "从总共 1M 到 15+ 路 × 1M：GLM-5.3 KV Cache 换出的容量突破"
  (From 1M total to 15+ x 1M: GLM-5.3 KV-cache offload).
* [ALG] "算法层：从注意力、KV Cache 到 FFN 与 MoE"
  (Algorithm layer: from attention and KV cache to FFN and MoE).
* [QNT] "量化不是压缩包：从模型分层到 4-bit 推理的工程真相"
  (Quantization is not a zip file).
* [W7] "双8卡(AMD W7900D)机器如何跑 GLM5.3"
  (How a dual 8-card AMD W7900D machine runs GLM5.3).

Modules:

* ``q8g64``     Q8G64 row layout and dequantisation.
* ``indexer``   DSA indexer scores and the Top-K selection.
* ``hotcache``  the GPU-managed hot cache, recent ring and write-back, as a
                sequential simulator with a position->slot index.
* ``naive_cache`` a second, deliberately naive simulator (linear scans, no
                index, per-miss hand walk) used only to pin ``hotcache``.
* ``attention`` absorbed-MLA decode attention over the selected rows.
* ``decode``    one decode step of one unit, composed from the above.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against brute force, closed forms, worked examples or invariants; none is
"parity unpinned".
"""
