"""fp64 CPU oracle for online-softmax attention and softmax -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference arm
may import this package.  The product library (``online_softmax_flash_gb300``) never
imports, links or calls it, and this package never imports the product: the two share no
code.  Inputs come from ``seeded_inputs`` (random draws only, no method arithmetic).

Sources, cited by page title and section:

* [SA] "softmax_attention" (blog.euler0525.cn/posts/3fb3592b): section "实现思路"
  (approach: the naive PyTorch ``solve``, the 32-key block loop, -inf tail masking, the
  running max / alpha / denominator / numerator recurrence and its pseudocode).
* [Q3] "从零开始写Qwen3（五-其一）使用Triton实现自注意力" (gitcode.csdn.net): sections
  "自注意力原理" (the torch GQA + causal definition), "softmax的triton实现", "多头自注意力",
  "GQA" (kv head = q head // group size).
* [TP] Triton-Puzzles write-up (fadingcoder.top/post/105980): "Puzzle 8: Long Softmax"
  (spec, "Brute-Force Approach (Three Loops)", "Optimized Approach (Two Loops with Online
  Softmax)"), "Puzzle 9: Simple FlashAttention".
* [SO] "Softmax 算子的实现与优化" (blog.euler0525.cn/posts/5db73590): "Triton 版本 ·
  Baseline" (three-stage stable softmax), "Online Softmax" (the boxed recurrence and its
  invariant), "CUDA 版本".

Every function here is pinned by a ``-m "not gpu"`` test against closed forms, brute
force, worked examples and invariants (``tests/test_oracle_pins.py``).
"""
from .attention import attention, attention_gqa, attention_rows
from .attention_bwd import attention_bwd, attention_gqa_bwd
from .softmax import softmax, softmax_masked
from .recurrence import (combine_partials, online_attention_row, online_softmax,
                         online_softmax_state)

__all__ = [
    "attention", "attention_gqa", "attention_rows", "attention_bwd", "attention_gqa_bwd", "softmax",
    "softmax_masked",
    "online_softmax_state", "online_softmax", "online_attention_row", "combine_partials",
]
