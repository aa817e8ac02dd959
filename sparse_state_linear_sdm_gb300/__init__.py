"""GB300 (sm_103a) Sparse Delta Memory forward hot path.

The compute lives in ``libsdm.so`` (CUDA C++, C ABI declared in include/sdm.h);
``api`` is a thin ctypes binding for torch tensors and ``workloads`` defines the
seeded synthetic configurations.  Importing the package does not load the
library; the first API call does (and fails loudly if it cannot).
"""
from .api import (BWD_DM0_ONLY, BWD_FINAL_ZERO, SELECT_AUTO, SELECT_COUNTING, SELECT_GENERAL, SDM_BF16, SDM_DEV_DUP_WRITE, SDM_DEV_INDEX_RANGE, SDM_DEV_TIMEOUT, SDM_F32, DecodeStep, SDMError,
                  backward_workspace_size, bounded_wait_check, copy_token_window, decode_step, decode_table, fill_state, forward,
                  forward_chunks, forward_workspace, scan_backward, scan_forward_train, select_backward,
                  gen_inputs, gen_M0, init_state_from_M0, lib, library_path, pinned_empty, project_kq, project_select, project_select_workspace,
                  project_stall_check, scan_forward,
                  scan_forward_noalloc, NOALLOC_SCRATCH_BYTES, scan_launch_info, scan_workspace, scan_workspace_size, select, side_stream)

__all__ = ["BWD_DM0_ONLY", "BWD_FINAL_ZERO", "SELECT_AUTO", "SELECT_COUNTING", "SELECT_GENERAL", "SDM_BF16", "SDM_DEV_DUP_WRITE", "SDM_DEV_INDEX_RANGE", "SDM_DEV_TIMEOUT", "SDM_F32", "DecodeStep", "SDMError",
           "backward_workspace_size", "bounded_wait_check", "copy_token_window", "decode_step", "decode_table", "fill_state", "forward",
           "forward_chunks", "forward_workspace", "scan_backward", "scan_forward_train", "select_backward",
           "gen_inputs", "gen_M0", "init_state_from_M0", "lib", "library_path", "pinned_empty", "project_kq", "project_select", "project_select_workspace",
           "project_stall_check", "scan_forward",
           "scan_forward_noalloc", "NOALLOC_SCRATCH_BYTES", "scan_launch_info", "scan_workspace", "scan_workspace_size", "select", "side_stream"]
