"""GB300-native blockwise online-softmax (Ring Attention forward) library.

The compute path is ``libra.so``, a C-ABI library of hand-written sm_103a
CUDA kernels.  ``binding`` marshals torch tensors into it.  Importing this
package does not load the library.  The first call of a binding function
loads it, and raises if it has not been built.
"""

from .binding import (  # noqa: E402,F401
    LAYOUTS,
    RaError,
    layout_positions,
    ra_block_update,
    ra_block_update_masked,
    ra_cached_memory,
    ra_decode_forward,
    ra_decode_partial,
    ra_device_status,
    ra_finalize,
    ra_merge,
    ra_release_cached_memory,
    ra_ring_forward,
    ra_ring_forward_host,
    ra_ring_forward_masked,
    ra_ring_backward,
    ra_ring_backward_masked,
    ra_ring_forward_noalloc,
    ra_ring_step,
    ra_ring_step_masked,
    ra_selftest_wait_timeout,
    ra_state_init,
    ra_trace_enable,
    ra_trace_query,
    ra_trace_reset,
)
