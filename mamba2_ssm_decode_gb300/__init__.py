"""GB300 (sm_103a) Mamba2 selective-state-update decode.

The C ABI lives in include/ssu.h and libssu_gb300.so (built in-tree by
``mamba2_ssm_decode_gb300.build``); this package binds it for CUDA torch
tensors:

  ssu_update         one-token decode step
  ssu_update_varlen  packed variable-length / speculative (MTP) step
  ssu_replay_update  ReplaySSM checkpointing update (ring caches, trackers)
  ssu_replay_update_static  the same for callers that cannot pass scratch memory
  ssd_combined_fwd_varlen  packed variable-length SSD prefill (chunk states)
  ssu_ring_update    ReplaySSM ring-tracker update or reset
  ssu_ring_commit    ReplaySSM ring-tracker commit of the previous window
  ssu_device_error   the device error word of the bounded waits (diagnostic)
  ssu_selftest_bounded_wait  proves on the device that a bounded wait gives up
"""
from .api import (ssd_combined_fwd_varlen, ssd_workspace_bytes, ssu_device_error,
                  ssu_replay_update, ssu_replay_update_static,
                  ssu_ring_commit, ssu_ring_update, ssu_selftest_bounded_wait, ssu_update,
                  ssu_update_varlen)

__all__ = ["ssu_update", "ssu_update_varlen", "ssu_replay_update", "ssu_replay_update_static",
           "ssu_ring_update", "ssu_ring_commit", "ssd_combined_fwd_varlen", "ssd_workspace_bytes",
           "ssu_device_error", "ssu_selftest_bounded_wait"]
