"""Plain, slow CPU oracle for the CSA / HCA forward pass, in float64.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product (the CUDA library under ``long_context_sparse_25_b300``
and its Python binding) never imports, links or calls anything here, and this
package imports nothing from the product.

Every function cites the passage of the pages it follows.  The pages are:

* "一文搞懂 DeepSeek：从 V3 的 KV 压缩与 MoE，到 V4 的百万 token 上下文"
  (deepseek.csdn.net) -- the most precise statement of CSA / HCA, section
  "V4 改进一：CSA 与 HCA", and the MLA description in section
  "V3 看家本领一：MLA".
* "DeepSeek-V4 详解" (yudonglee.me) -- section 2.2 (CSA Steps 1-4) and
  section 2.3 (HCA Steps 1-2).
* "DeepSeek-V4 — 百万 Token 上下文的高效 MoE 模型" (jaylab-temp.pages.dev) --
  the bullets on RMSNorm of queries / KV entries and on the mixed BF16/FP8
  KV cache.
* the hongke120.com page on DeepSeek-V4 (its text carries no title) --
  sections 2.2 / 2.3 (CSA / HCA overview; read where it agrees with the two
  pages above).

Parity status: every function in ``csa_oracle`` is pinned by a ``-m "not gpu"``
test in ``tests/test_oracle_pins.py`` except the full composition at the large
workloads, which has no closed form; there the pins on each step and the
brute-force composition on tiny inputs are what stands behind it.
"""

from .csa_oracle import *  # noqa: F401,F403
