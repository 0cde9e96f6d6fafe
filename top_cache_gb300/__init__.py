"""GB300-native sparse-decode KV offload hot path (libkvo + its Python binding)."""
from .kvo import (  # noqa: F401
    EXPORTED, KVO_ECAPACITY, KVO_ECUDA, KVO_EINVAL, KVO_ENOMEM, KVO_ERANGE, KVO_ETIMEOUT,
    KVO_GATHER_BULK, KVO_GATHER_LDG, KVO_OK, KVO_OPT_GATHER_MODE, KVO_OPT_GROUPS, KVO_OPT_PROFILE, KVO_OPT_SCORE_CTAS, KVO_OPT_SPECULATE, KVO_OPT_WAIT_LIMIT_NS, PROF_KINDS,
    KVO_PAD_PAYLOAD, Kvo, KvoError, kvo_append, kvo_create, kvo_destroy, kvo_export_state,
    kvo_get_stats, kvo_host_rows, kvo_prefill, kvo_profile_read, kvo_reset, kvo_select, kvo_select_noalloc, kvo_select_workspace_size,
    kvo_set_option, kvo_step, lib, library_path,
)
