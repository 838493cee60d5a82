"""B300-native (sm_103a) selective scan of the Mamba selective state-space model.

Public calls (thin wrappers over the C ABI in include/ssm_scan.h):

* ``ssm_scan_fwd``     -- full-sequence scan (prefill / training forward);
* ``ssm_state_update`` -- single-token recurrent update (decode).

The CUDA library ``libssmscan.so`` is loaded on first use; there is no CPU
fallback.
"""
from ._lib import (SSMError, device_error, load_library, scan_workspace_bytes,  # noqa: F401
                   ssm_scan_fwd, ssm_state_update, status_string)

__all__ = ["ssm_scan_fwd", "ssm_state_update", "scan_workspace_bytes", "device_error",
           "load_library", "status_string", "SSMError"]
