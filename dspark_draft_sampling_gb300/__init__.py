"""libdspark: GB300-native DSpark per-cycle draft step (Markov block draft,
Q8_0 confidence probe, weight-stationary small-M matvec).

Every step of the path runs in the CUDA kernels of ``libdspark.so``; this package
only marshals torch tensors into the C ABI declared in ``include/dspark.h``.
"""
from .api import (  # noqa: F401
    DraftPlan,
    DsparkError,
    GatedDraftPlan,
    MarkovPlan,
    ProbeCall,
    conf_probe,
    conf_probe_host,
    conf_probe_split,
    lib_path,
    load_library,
    markov_draft,
    markov_draft_host,
    markov_workspace_bytes,
    q8_0_repack,
    ws_matvec,
    ws_matvec_grouped,
    ws_matvec_host,
    ws_matvec_q8,
    ws_matvec_q8_workspace_bytes,
    ws_matvec_workspace_bytes,
)
