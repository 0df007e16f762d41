"""CPU oracle for the Falcon fast-weight forward (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU baseline
legs may import this package.  It shares no code with the CUDA library.
"""

from .falcon import (  # noqa: F401
    FALCON_1, FALCON_1A, FALCON_2, FALCON_2A, FALCON_3, FALCON_3A, VARIANT_NAMES,
    build_pairs, chunked, decay_factor, effective_window, is_additive,
    is_per_channel, is_windowed, masked_parallel, recurrent, recurrent_heads,
    step_coefficients,
)
from .falcon_grad import ONE_PAIR, recurrent_torch, recurrent_vjp  # noqa: F401,E402
from .prologue import GATE_LOGITS, L2NORM_QK, apply_prologue, phi, recurrent_varlen, sigmoid  # noqa: F401,E402
