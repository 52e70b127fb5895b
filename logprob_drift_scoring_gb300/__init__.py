"""Selected-token logprob drift scoring on one GB300 (sm_103a).

The computation lives in liblpd.so (C ABI, include/lpd.h), built from the
CUDA sources in csrc/.  ``binding`` is its thin Python binding (same names,
argument marshalling only); ``workloads`` holds the seeded synthetic inputs.
"""
from .binding import (  # noqa: F401
    LpdError,
    lpd_backend_info,
    lpd_drift_metrics,
    lpd_score,
    lpd_score_sharded,
    lpd_select_active,
    lpd_strerror,
    lpd_token_logp,
    lpd_workspace_size,
    read_metrics,
    score,
)
