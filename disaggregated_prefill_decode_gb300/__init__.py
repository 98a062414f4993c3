"""kvx: paged KV-cache push between two pools in one GPU's HBM (sm_103a), with a C-ABI (include/kvx.h).

``from disaggregated_prefill_decode_gb300 import kvx`` loads libkvx.so and exposes the C calls under
their own names (kvx_plan, kvx_push_layer, kvx_sync, kvx_match_prefix, ...).
"""
