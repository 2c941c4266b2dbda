"""GB300 (sm_103a) OSDN forward path: phase-1 preconditioner scan, chunkwise preconditioned
delta rule, and single-token decode, behind the C ABI of include/osdn.h.

The CUDA library (libosdn.so) is loaded on first use; a missing library raises ImportError.
"""
from .binding import (OSDN_BF16, OSDN_F16, OSDN_F32, OsdnError, chunk_osdn, osdn_check,
                      osdn_chunk_fwd, osdn_chunk_fwd_workspace_bytes, osdn_decode_step, osdn_layer_fwd,
                      osdn_layer_bwd, osdn_layer_bwd_workspace_bytes,
                      osdn_layer_fwd_host, osdn_layer_fwd_host_workspace_bytes,
                      osdn_layer_fwd_varlen, osdn_layer_fwd_varlen_workspace_bytes,
                      osdn_layer_fwd_workspace_bytes, osdn_precond_scan, osdn_precond_scan_workspace_bytes,
                      osdn_status_string,
                      osdn_version)

__all__ = ["OSDN_BF16", "OSDN_F16", "OSDN_F32", "OsdnError", "chunk_osdn", "osdn_check",
           "osdn_chunk_fwd", "osdn_chunk_fwd_workspace_bytes", "osdn_decode_step", "osdn_layer_fwd",
           "osdn_layer_bwd", "osdn_layer_bwd_workspace_bytes",
           "osdn_layer_fwd_host", "osdn_layer_fwd_host_workspace_bytes",
           "osdn_layer_fwd_varlen", "osdn_layer_fwd_varlen_workspace_bytes",
           "osdn_layer_fwd_workspace_bytes", "osdn_precond_scan", "osdn_precond_scan_workspace_bytes",
           "osdn_status_string",
           "osdn_version"]
