"""libfattn for NVIDIA GB300 (sm_103a): exact attention forward with the
online-softmax recurrence, and row-wise online softmax / log-sum-exp.

The compute path is the C-ABI library ``libfattn.so`` (include/fattn.h), built
in-tree by :mod:`online_softmax_10_gb300.build`; :mod:`.fattn` is its thin
binding.  :mod:`.inputs` holds the seeded synthetic input generators.
"""
from .fattn import (FattnError, attn_fwd, attn_fwd_splitkv, attn_fwd_strided, cross_entropy_rows,  # noqa: F401
                    device_status,
                    log_softmax_rows, logsumexp_rows,
                    selftest_wait_timeout, softmax_rows, splitkv_num_splits, splitkv_workspace_bytes,
                    status_string, version)
