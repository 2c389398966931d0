"""Context-parameter clamps.

UBATCH, section "Three things called batch": n_batch is the logical limit on
one decode call, n_ubatch the physical size of one forward pass.  At context
creation the physical size is clamped to the logical one, and under causal
attention the logical size is itself clamped to the cache capacity n_ctx.
A requested n_ubatch of 0 means "same as n_batch".  Defaults (UBATCH, section
"Back to the VRAM question"; BATCH-ZH, section "两级批次参数"): n_batch 2048,
n_ubatch 512.
"""

DEFAULT_N_BATCH = 2048
DEFAULT_N_UBATCH = 512


def clamp(n_ctx, n_batch, n_ubatch, causal):
    """Return the effective (n_batch, n_ubatch).

    UBATCH, "Three things called batch": under causal attention the caller
    cannot submit more positions than the cache holds, so n_batch becomes
    min(n_ctx, n_batch); non-causal models keep the requested n_batch.  The
    effective n_ubatch is then the smaller of that n_batch and the request
    (the request 0 standing for n_batch).
    """
    if causal:
        eff_batch = min(n_ctx, n_batch)
    else:
        eff_batch = n_batch
    requested_ubatch = n_batch if n_ubatch == 0 else n_ubatch
    eff_ubatch = min(eff_batch, requested_ubatch)
    return eff_batch, eff_ubatch
