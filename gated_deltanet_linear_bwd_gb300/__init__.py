"""Gated DeltaNet chunked prefill (forward + backward) for one GB300 (sm_103a).

The computation runs in libgdn.so (C ABI in include/gdn.h); this package is
its thin Python binding.  Importing it loads the library and fails loudly if
it has not been built.
"""
from . import _abi
from ._abi import (GDN_BF16, GDN_CP_AUTO, GDN_CP_FORCE, GDN_CP_OFF, GDN_FP32, GdnError,
                   gdn_abi_version, gdn_bwd_workspace_size, gdn_chunk_bwd, gdn_chunk_fwd,
                   gdn_fwd_ctx_size, gdn_fwd_workspace_size, gdn_last_error, gdn_profile_begin, gdn_profile_end,
                   gdn_recurrent_step, gdn_set_spin_limit, gdn_sync_status)
from .api import (chunk_gated_delta_rule, chunk_gated_delta_rule_bwd,
                  chunk_gated_delta_rule_fwd, recurrent_step)

_abi.load()

__all__ = ["chunk_gated_delta_rule", "chunk_gated_delta_rule_fwd", "chunk_gated_delta_rule_bwd",
           "recurrent_step", "gdn_recurrent_step",
           "gdn_abi_version", "gdn_fwd_workspace_size", "gdn_fwd_ctx_size", "gdn_chunk_fwd",
           "gdn_bwd_workspace_size", "gdn_chunk_bwd", "gdn_sync_status", "gdn_last_error",
           "gdn_set_spin_limit", "gdn_profile_begin", "gdn_profile_end", "GdnError", "GDN_FP32", "GDN_BF16", "GDN_CP_AUTO",
           "GDN_CP_OFF", "GDN_CP_FORCE"]
