"""fp64 CPU oracle (test infrastructure only; never imported by the library).

See oracle/attention.py for what each function computes and which passage of
the pages it follows.  Parity is pinned for every function here except the
hand-worked example of "Transformer 与 LLM" slide 01 (its inputs are not
printed: parity unpinned, only the row-sum property is checked).
"""
from .attention import (  # noqa: F401
    NEG_INF,
    attention_decode,
    attention_head,
    attention_prefill,
    attention_prefill_rows,
    causal_mask,
    default_scale,
    logsumexp_rows,
    mla_absorb_query,
    mla_decode_unabsorbed,
    mla_prefill_unabsorbed,
    mla_unabsorb_output,
    rope_cache,
    rope_frequencies,
    rope_rotate,
    softmax_rows,
)
