"""GB300-native hybrid optimizer step: batched Muon on view-split 2-D weights
plus the clipped AdamW path, as a C-ABI CUDA library with a ctypes binding.

The library (``_lib/libgbo.so``) is built by :func:`build.build`.  The
binding functions carry the names of the C entry points in ``include/gbo.h``.
"""

from ._binding import (  # noqa: F401
    GBO_BF16, GBO_F32, GBO_NS_BF16, GBO_NS_F32, GBO_STATUS_NONFINITE, GBO_STATUS_TIMEOUT,
    GboError, MuonPlan, PHASE_NAMES,
    gbo_abi_version, gbo_adamw_step, gbo_clip_norm, gbo_clip_norm_noalloc, gbo_clip_norm_workspace_bytes,
    gbo_desc_hash, gbo_h2d_copy,
    gbo_last_error, gbo_launch_count, gbo_muon_plan_create, gbo_muon_plan_destroy,
    gbo_muon_plan_info, gbo_muon_plan_phase_times, gbo_muon_plan_set_event, gbo_muon_plan_set_free_sms,
    gbo_muon_plan_set_stats, gbo_muon_plan_set_timing,
    gbo_muon_step,
    gbo_muon_workspace_bytes, gbo_normuon_rownorm, gbo_struct_size, lib, library_path,
)
