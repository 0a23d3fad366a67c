"""CPU oracle for the MXFP8 decode-step hot path -- TEST INFRASTRUCTURE ONLY.

A plain, slow, fp64 numpy restatement of what the hot path computes, written
from the pages' statement of the method (cited per function, by page title and
section). It shares no code with the CUDA path and imports nothing from it.
Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import it; the product path never
routes through it.

Pages cited (by title):

* [S2.1] "How We Made Our Text-to-Speech API Free: The Inference Engineering
  Behind S2.1 Pro" (Fish Audio engineering post; also published in Chinese as
  "我们如何实现文本转语音 API 免费：S2.1 Pro 背后的推理工程"), sections
  "FP8 Quantization Strategy", "Kernel Benchmark Results",
  "DualAR: S2-Specific Batching Constraints", "What's Open Source".
* [FSKV] "Fish Speech KV Cache 推理优化记录" (Fish Speech PR #1312 write-up),
  §4 "瓶颈：有因果 mask，仍然传入了完整缓存", §5 "修改：保留容量，只读取 active
  prefix", §7 "Review：加速之外，还要定义正确性".

The MX element/scale rules are not printed on the pages beyond "1x32 blocks,
E4M3 elements, OCP UE8M0 shared exponents"; ``oracle.mx`` follows the public
OCP Microscaling Formats (MX) v1.0 specification for the missing steps.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against hand-worked values, closed forms, library routines (torch float8
casts, torch SDPA, torch rms_norm) or brute force. No function is "parity
unpinned".
"""
from . import mx, ops  # noqa: F401
