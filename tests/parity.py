"""Shared helpers of the GPU parity tests: run the oracle on a host step and
compare the CUDA results with it."""

import numpy as np

import oracle

# |gpu - oracle| <= max(ABS_TOL, REL_TOL * |oracle|) per element: bf16 inputs,
# fp32 accumulation, bf16 output against an fp64 oracle.
ABS_TOL = 2e-2
REL_TOL = 1e-2


def bits_to_f64(bits):
    return oracle.bf16_bits_to_f64(bits)


def oracle_step(step, rows=None):
    """Oracle slot mapping, post-write pool and attention output (fp64)."""
    slots = oracle.slot_mapping(step.block_table, step.query_start_loc, step.num_computed,
                                step.block_size)
    pool = oracle.kv_write(step.kv_cache, step.k, step.v, slots)
    out = oracle.paged_attention(step.q, pool, step.block_table, step.seq_lens,
                                 step.query_start_loc, step.num_computed, step.scale, rows=rows)
    return slots, pool, out


def assert_close(gpu_bits, ref, rows=None, what="attention"):
    """Element-wise tolerance check of bf16 GPU output against the fp64 oracle."""
    g = bits_to_f64(gpu_bits)
    if rows is not None:
        g, ref = g[rows], ref[rows]
    assert np.isfinite(ref).all(), "oracle output has non-finite values"
    err = np.abs(g - ref)
    bound = np.maximum(ABS_TOL, REL_TOL * np.abs(ref))
    bad = ~(err <= bound)  # NaN in g counts as bad
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; "
            f"max abs err {np.nanmax(err):.3e}; first bad {idx.tolist()} "
            f"gpu={g[tuple(idx[0])]} ref={ref[tuple(idx[0])]}")
    return float(err.max()), float((err / np.maximum(np.abs(ref), ABS_TOL / REL_TOL)).max())
