"""B300-native (sm_103a) selective scan of the Mamba selective state-space model.

Public calls (thin wrappers over the C ABI in include/ssm_scan.h):

* ``ssm_scan_fwd``     -- full-sequence scan (prefill / training forward);
* ``ssm_state_update`` -- single-token recurrent update (decode).

The CUDA library ``libssmscan.so`` is loaded on first use; there is no CPU
fallback.
"""
from ._lib import (SSMError, load_library, ssm_scan_fwd, ssm_state_update,  # noqa: F401
                   status_string)

__all__ = ["ssm_scan_fwd", "ssm_state_update", "load_library", "status_string", "SSMError"]
