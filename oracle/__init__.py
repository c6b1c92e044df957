"""CPU oracle (test infrastructure). See ``oracle.paged_attention``."""
from .paged_attention import (attend_row, attention, default_scale, gather,  # noqa: F401
                              kv_bytes_per_token, kv_head_of, row_weights,
                              slot_location, softmax_weights, visible_keys,
                              widen, write_kv)
