"""CPU oracle for the kvtc hot path (TEST INFRASTRUCTURE ONLY).

A plain, slow, fp64 NumPy restatement of KV-cache transform coding as the
page "KV Cache Transform Coding for Compact Storage in LLM Inference"
(gist.science summary of arXiv 2511.01815, Technical summary section 2
Methodology, parts A Calibration, B Compression, C Decompression) describes
it.  It exists to check the CUDA path and nothing else:

* only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
  ``bench.py`` may import it;
* it shares no code with the CUDA path (``kv_cache_transform_gb300``), and
  neither imports the other;
* its inputs come from ``synth`` (seeded draws, no codec arithmetic) or from
  its own functions, never from the CUDA path.

Modules:
  fp         -- IEEE binary16 round-down / round-up / nearest and bf16 nearest
                from fp64, written from the format definitions.
  codec      -- microscaled quantiser, bit-plane record packing, stream
                compress / decompress / paged decompress.
  calibrate  -- PCA basis, measured distortion table, DP bit allocation,
                calibration blob writer.
  fieldpack  -- lossless field packing of a stream's records (the sign and
                exponent of each fp16 field as an offset from the stream's
                minimum), our stand-in for the page's entropy stage.

Parity status: every function is pinned by ``tests/test_oracle_*.py``
(brute force, closed forms, invariants, library special cases).  The one
thing not pinned is the quality of the bit allocation against the page's
accuracy results (that needs trained models and datasets): parity unpinned
versus the paper's accuracy numbers.
"""
