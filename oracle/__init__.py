"""CPU oracle for the fused attention forward — TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The
product path (``exact_attention_86_gb300``) never imports it and has no CPU
fallback: if the CUDA library is missing, the product raises.

Contents:

* ``attention.attention_ref`` — the plain definition of exact attention,
  ``softmax(Q K^T * scale + mask) V`` with the per-row log-sum-exp, in float64,
  with every score row materialised in full ("Kernel Fusion and the Memory
  Wall", section "FlashAttention: avoid the full score matrix"; the stable
  softmax of section "Softmax needs a global row statistic").
* ``attention.attention_rows`` — the same definition for a chosen set of query
  rows of one head, used for sampled parity at full size.
* ``attention.attention_varlen_ref`` — the same definition for a packed batch
  of variable-length sequences (each sequence on its own tokens).
* ``attention.attention_paged_ref`` — packed queries against a paged key/value
  cache: each sequence's keys gathered through its page table, then the same
  definition.
* ``fp8.decode_e4m3`` / ``fp8.attention_fp8_ref`` — E4M3 codes decoded from
  the format definition, and exact attention of FP8 inputs with per-tensor
  descales.
* ``backward.attention_bwd_ref`` (and ``attention_bwd_head``,
  ``attention_bwd_sampled``) — gradients of the forward with respect to Q, K
  and V for an upstream dO, from the chain rule on the materialised softmax.
* ``online.online_softmax_attention`` — the tiled online-softmax recurrence
  (running max, normaliser, numerator, each corrected by exp(m_old - m_new))
  from "Attention softmax fusion", section "The tile loop", and "Kernel Fusion
  and the Memory Wall", section "FlashAttention: avoid the full score matrix".
  It exists only so the tests can pin the materialised form against it.
* ``merge.lse_merge`` — the combination of per-key-range partial results
  (normalised partial output and LSE of each range) into the whole-row result.

The oracle shares no code with the CUDA path: it reads float64 NumPy arrays
and nothing else.
"""

from .attention import (attention_paged_ref, attention_ref, attention_rows, attention_varlen_ref,  # noqa: F401
                        valid_key_count)
from .online import online_softmax_attention  # noqa: F401
from .merge import lse_merge  # noqa: F401
from .fp8 import attention_fp8_ref, decode_e4m3  # noqa: F401
from .backward import attention_bwd_head, attention_bwd_ref, attention_bwd_sampled  # noqa: F401
