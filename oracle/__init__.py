"""fp64 CPU oracle (test infrastructure; see ``splash_oracle``)."""
from .splash_oracle import (PagedPool, accept_commit, attention, attention_partial, attention_seq_head,  # noqa: F401
                            dequantise, gather_keys, kv_append, lse_combine, quantise_rows)
