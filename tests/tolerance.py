"""Comparison rules shared by the parity tests.

Attention outputs are f16 computed with f32 accumulation; an element passes
when ``|gpu - ref| <= ATOL + RTOL * |ref|`` with ATOL = 2e-3 and RTOL = 1e-2
(max-abs 2e-3 / max-rel 1e-2, read as an allclose bound).  Append is compared
bit for bit.
"""

import numpy as np

ATOL = 2e-3
RTOL = 1e-2


def attention_errors(gpu, ref):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    diff = np.abs(gpu - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = ~(diff <= bound)  # NaN counts as bad
    rel = diff / np.maximum(np.abs(ref), 1e-30)
    return {
        "max_abs": float(np.nanmax(diff)) if diff.size else 0.0,
        "max_rel_where_ref_gt_0.1": float(np.nanmax(np.where(np.abs(ref) > 0.1, rel, 0.0))) if diff.size else 0.0,
        "n_bad": int(bad.sum()),
        "n": int(diff.size),
        "first_bad": tuple(int(i) for i in np.argwhere(bad)[0]) if bad.any() else None,
    }


def assert_attention_close(gpu, ref, what=""):
    e = attention_errors(gpu, ref)
    assert e["n_bad"] == 0, f"{what}: {e}"
    return e


def assert_bits_equal(a, b, what=""):
    a16 = np.ascontiguousarray(a).view(np.uint16)
    b16 = np.ascontiguousarray(b).view(np.uint16)
    assert a16.shape == b16.shape, what
    neq = a16 != b16
    assert not neq.any(), f"{what}: {int(neq.sum())} differing f16 words, first at {np.argwhere(neq)[0]}"
