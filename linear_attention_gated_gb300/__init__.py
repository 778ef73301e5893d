"""GB300 (sm_103a) recurrent KDA training forward + backward behind a C ABI.

``kda_fwd`` / ``kda_bwd`` (and the aliases ``recurrent_kda_training_forward`` /
``recurrent_kda_training_backward``), the standalone ``recurrent_kda_backward``
(with a reusable ``RecurrentKDABackwardWorkspace``), the inference
``kda_prefill`` and the single-token ``kda_decode`` call libkda.so; ``HostStep`` runs whole training
steps from and to host memory (``kda_step_host``); see include/kda.h.
"""

from .kda import (  # noqa: F401
    EXPORTED,
    GRAD_NAMES,
    HostStep,
    KdaContext,
    KdaError,
    RecurrentKDABackwardWorkspace,
    kda_bwd,
    kda_bwd_noalloc,
    kda_decode,
    kda_fwd,
    kda_prefill,
    load_library,
    noalloc_status,
    recurrent_kda_backward,
    recurrent_kda_training_backward,
    recurrent_kda_training_forward,
    workspace_bytes,
)
