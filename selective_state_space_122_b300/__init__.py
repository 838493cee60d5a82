"""B300-native (sm_103a) selective scan of the Mamba selective state-space model.

Public calls (thin wrappers over the C ABI in include/ssm_scan.h):

* ``ssm_scan_fwd``     -- full-sequence scan (prefill / training forward),
                          optionally from an initial state (``initial_state=``);
                          B and C shaped (batch, ngroups, N, L) give every group
                          of dim / ngroups channels its own B and C (also for
                          ``ssm_state_update`` and ``ssm_scan_bwd``);
* ``ssm_state_update`` -- single-token recurrent update (decode);
* ``ssm_scan_bwd``     -- the scan's backward (every input's gradient);
* ``conv1d_fwd``       -- the depthwise causal conv1d (+ SiLU) that produces the
                          scan input, with a carried conv state;
* ``conv1d_update``    -- its single-token decode step.

The CUDA library ``libssmscan.so`` is loaded on first use; there is no CPU
fallback.
"""
from ._lib import (SSMError, conv1d_fwd, conv1d_update, device_error, force_scan_path,  # noqa: F401
                   load_library, scan_workspace_bytes, ssm_scan_bwd, ssm_scan_fwd, ssm_state_update,
                   status_string)

__all__ = ["ssm_scan_fwd", "ssm_state_update", "ssm_scan_bwd", "conv1d_fwd", "conv1d_update", "scan_workspace_bytes",
           "device_error", "force_scan_path", "load_library", "status_string", "SSMError"]
