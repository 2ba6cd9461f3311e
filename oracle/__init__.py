"""CPU oracle (test infrastructure only; see ``attn_ref``)."""
from .attn_ref import (  # noqa: F401
    attention, attention_rows, attention_bruteforce, probabilities,
    online_softmax_attention, rebase_threshold_in_other_units, LOG2E, LN2,
)
