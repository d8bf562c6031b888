"""GB300-native vocab-parallel LM-head logits gather on a two-parity Lamport
mailbox, for TP virtual ranks on one GPU.

The library is libhg.so (C ABI in include/hg.h, CUDA kernels for sm_103a);
``hg`` is its Python binding and ``synth`` makes seeded synthetic inputs.
"""

from . import hg, synth  # noqa: F401
from .hg import (GatherCall, HGError, Handle, hg_create, hg_debug_skip_push,  # noqa: F401
                 hg_destroy, hg_gather, hg_gather_fused, hg_gather_host, hg_gather_static,
                 hg_gather_stats, hg_launch_shape, hg_mailbox, hg_parity, hg_rearm,
                 hg_stock_gather, hg_sync, mailbox_words, new_row_stats, unpack_row_stats)
