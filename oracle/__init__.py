"""CPU oracle for the NVFP4 sparse-MLA pack and decode calls.

TEST INFRASTRUCTURE ONLY. This package is the plain, slow, obviously correct
restatement of what the CUDA path computes, written in numpy float64 from the
source pages. Only the test suite, ``__graft_entry__.smoke()`` and the CPU
baseline / reference arm of ``bench.py`` may import it. The library itself
(``nvfp4_sparse_mla_gb300``) never imports, links or calls anything here, and
nothing here imports the library: the two share no code, tables or constants.
Inputs come from ``nvfp4_sparse_mla_gb300.workloads`` (random numbers and
layout only).

Sources (web pages, cited by title and section):

* "Prime Inference: Fast, Reliable Serving for Frontier Open Models"
  (devoured.fyi digest), sections "Making room for low-latency decode" and
  "A native NVFP4 sparse-MLA decode kernel".
* "Prime Inference open-model serving" (mo.ai.kr news), section
  "KV 캐시와 데이터 전송" (KV cache and data transfer).
* "Prime Intellect unveils Prime Inference" (wireai.ir), section
  "4-bit caches open the way", items 1-3.

Modules:

* ``formats``   -- E2M1 and E4M3 code tables, decode and round-to-nearest-even
                   encode (pinned).
* ``pack``      -- the 352-byte cache row writer (pinned).
* ``attention`` -- masked sparse softmax attention over selected rows (pinned).
* ``staged``    -- the staged baseline's FP8 requantisation (pinned).
* ``layered``   -- one layer of a block-major multi-layer cache (pinned).
* ``fp8cache``  -- the 576-byte FP8 cache and its decode (pinned).
* ``topk``      -- the -1 padded top-k lists (pinned).

Every function is pinned by tests under ``tests/`` against facts the pages
or mathematics fix (printed grid and byte counts, library conversions,
closed forms, brute force); none is marked "parity unpinned".
"""

from . import formats, pack, attention, staged  # noqa: F401
