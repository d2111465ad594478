"""Context-parallel Gated DeltaNet forward for one GB300 (sm_103a).

The computation lives in the CUDA library ``libgdncp.so`` (C ABI declared in
``include/gdn_cp.h``); ``binding`` is its thin Python front end.
"""
from .binding import (GdnError, decode_plan, gdn_chunk_fwd, gdn_chunk_summary,  # noqa: F401
                      gdn_conv_silu, gdn_cp_plan, gdn_layer_fwd, gdn_shard_fwd, gdn_state_combine, load,
                      plan_words, shard_fwd_workspace_size, shard_fwd_workspace_min_size)
from .binding import chunk_bwd_workspace_size, gdn_chunk_bwd  # noqa: F401
