"""GB300-native Mamba-2 selective-state library: decode, chunked scan, and
speculative verify (state copies or ReplaySSM replay), behind the C ABI of
``include/ssm_state.h``.

Importing this package loads ``_lib/libssmstate.so`` (built by
``hybrid_serving_mamba_gb300.build.build()``); there is no CPU fallback.
"""
from ._binding import *  # noqa: F401,F403
from ._binding import EXPORTS, LIB_PATH, Pool, SSMError, library, make_config, ssm_config, ssm_slot_meta, status_string  # noqa: F401
from ._binding import ssm_receipt, ssm_stream_identity, stream_identity  # noqa: F401
from ._binding import GdnPool, make_gdn_config, ssm_gdn_config  # noqa: F401
