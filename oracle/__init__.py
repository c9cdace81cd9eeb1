"""CPU oracle of the displaced-patch layer step: TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously correct restatement of what the hot path computes (numpy
fp64, plus exact fp32 C for the refresh).  Only the tests, the smoke check and
the bench's CPU-baseline leg may import it; the product path never does, and it
shares no code with the CUDA library.

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, library routines, brute force, hand-worked golden cases).  The
absolute end-to-end image quality of the method (seams, FID) is "parity
unpinned": it needs trained weights and datasets that are not available.
"""
from .layer import (SYNC, STALE, GN_SPLICED, GN_SYNC, GN_PREVIOUS, round_bf16, to_storage, patch_rows, gn_partial_stats,  # noqa: F401
                    gn_apply_spliced, halo_conv3x3, linear, stale_kv_attention,
                    refresh_residual, apply_residual, halo_segments, layer_forward, layer_state_update,
                    patch_layer_step, empty_state)


def build() -> None:
    """Compile the C part of the oracle (building the checker is not using it)."""
    from . import refresh
    refresh.build()
