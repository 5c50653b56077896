"""CPU oracle for the exact attention forward pass and its gradient.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports, links or runs this
package: only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use it. It shares no code with the CUDA path, and it imports nothing
from the product package.

Pages cited in this package (by title and section):

* [HW-FA]  "手写 FlashAttention:拆开 SDPA 这个黑盒" (Hand-written FlashAttention),
           learn-llm.fim.ai chapter 19, steps ①–⑤.
* [FA-tiling] "FlashAttention 核心思路解析" (FlashAttention core ideas), ijyty.com,
           §1–§5.2.
* [KCS]    "内核案例研究：Flash Attention", the cnblogs translation of
           "Kernel case study: Flash Attention" (towardsdatascience).
"""

from .naive import (  # noqa: F401
    attention,
    attention_backward,
    attention_backward_cols,
    attention_backward_head,
    attention_backward_magnitudes,
    attention_backward_rows,
    attention_general,
    attention_general_head,
    attention_rows,
    general_mask,
    merge_partials,
    online_softmax_trace,
    online_weighted_sum,
    safe_softmax,
    scores,
)
