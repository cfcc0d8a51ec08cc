"""Float64 CPU oracle for the fused attention forward.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import, call or
execute this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code, header, table or constant with the CUDA path.

What it computes is the plain definition of attention that the pages say
FlashAttention reproduces exactly:

* "Ascend C advanced practice: a high-performance FlashAttention-2-style
  tile-level fused attention operator", section 1.1 (the three-step MHA
  definition: scores, softmax, weighted sum of V) and section 1.2 (the
  online-softmax identity O_i = sum_j e^{P_ij - m_i} V_j / l_i);
* "FlashAttention under the catlass template" (lnwmold news page), section
  "Principle", which states that the blocked result is mathematically equal
  to standard attention;
* "FlashAttention extreme optimisation on Ascend NPUs: from principle to
  practice", section "The core idea of FlashAttention: IO-aware"
  (``standard_attention``: matmul, softmax over the last axis, matmul).

``paged.py`` gathers a sequence's keys and values from a paged cache (the
first page's section 9) and applies the same definition to them.
``backward.py`` gives the gradients of that definition with respect to Q, K
and V (the chain rule through it), for the backward pass the second page
says the operator also has.  ``rope.py`` adds the rotary position embedding that the first page's
section 9 ("Extensions: integration with RoPE and a paged KV cache") says
is applied to the Q and K blocks as they are loaded.

Every function here is pinned by ``tests/test_oracle.py`` against something
other than itself (brute force in exact arithmetic, closed forms, invariants,
a foreign library).  No function is "parity unpinned".
"""

from .attention import (  # noqa: F401
    MASK_NONE,
    MASK_CAUSAL,
    MASK_WINDOW,
    allowed_mask,
    attention_probs,
    attention_three_pass,
    attention_grouped,
    attention_online,
    attention_bruteforce,
    unmasked_pairs,
)
from .backward import attention_backward, attention_backward_grouped, attention_backward_sampled  # noqa: F401
from .paged import attention_paged, gather_pages  # noqa: F401
from .rope import (  # noqa: F401
    STYLE_HALF,
    STYLE_INTERLEAVED,
    apply_rope,
    attention_rope,
    pair_index,
    rope_tables,
)
