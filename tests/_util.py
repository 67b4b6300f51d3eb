"""Shared helpers of the parity tests: run the oracle and the library on one workload and
compare them with the step's acceptance rules."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from gqa_decode_attention_fa_gb300.workloads import Workload, bits, ints

# The step's acceptance tolerance on the bf16 output against the fp64 oracle.
MAX_ABS = 1e-2
REL_L2 = 2e-3

# A binary64 k row differs from the oracle's only if the exact value lies this close
# (relative) to a bf16 rounding midpoint; the rotated q rows are binary32, which moves the
# value by at most ~2^-20 of |y_i| + |y_partner| (norm scalar, cos/sin rounding, one fma).
K_MIDPOINT_WINDOW = 2.0 ** -40
Q_MIDPOINT_WINDOW = 2.0 ** -18


def geom_of(w: Workload):
    return oracle.geom(w.B, w.Hq, w.Hkv, w.d, w.block_size, w.max_seq, w.num_rows)


def oracle_step(w: Workload, pairs=None, threads=None):
    return oracle.decode_step(geom_of(w), bits(w.q_new), bits(w.k_new), bits(w.v_new), bits(w.k_cache),
                              bits(w.v_cache), ints(w.page_table), ints(w.seq_lens), ints(w.positions),
                              bits(w.q_norm_w), bits(w.k_norm_w), w.rope_theta, w.eps, pairs=pairs,
                              threads=threads)


def out_errors(gpu_bf16: torch.Tensor, ref: np.ndarray):
    g = gpu_bf16.float().cpu().double().numpy().reshape(ref.shape)
    diff = g - ref
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    rel = float(np.linalg.norm(diff) / max(np.linalg.norm(ref), 1e-300))
    return max_abs, rel


def assert_out_close(gpu_bf16, ref, what=""):
    max_abs, rel = out_errors(gpu_bf16, ref)
    assert np.all(np.isfinite(gpu_bf16.float().cpu().numpy())), f"{what}: non-finite output"
    assert max_abs <= MAX_ABS and rel <= REL_L2, f"{what}: max_abs={max_abs:.3e} rel_l2={rel:.3e}"
    return max_abs, rel


def _midpoint_distance(z: np.ndarray, got_bits: np.ndarray, want_bits: np.ndarray):
    """For elements whose bf16 bits differ: |z - m| where m is the midpoint between the two
    (adjacent) bf16 values; inf if the two values are not adjacent."""
    gv = torch.from_numpy(got_bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    wv = torch.from_numpy(want_bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    adjacent = np.abs(got_bits.astype(np.int64) - want_bits.astype(np.int64)) == 1
    mid = 0.5 * (gv + wv)
    return np.where(adjacent, np.abs(z - mid), np.inf)


def rotated_rows(w: Workload, which: str):
    """Exact (fp64) RMSNorm+RoPE values of the new q or k rows from the oracle's own
    building blocks, and the per-element slack scale |y_i| + |y_partner|."""
    src = bits(w.q_new if which == "q" else w.k_new).reshape(w.B, -1, w.d)
    wt = bits(w.q_norm_w if which == "q" else w.k_norm_w)
    wd = None if wt is None else oracle.bf16_to_f64(wt)
    pos = ints(w.positions)
    z = np.zeros(src.shape)
    scale = np.zeros(src.shape)
    for b in range(src.shape[0]):
        for h in range(src.shape[1]):
            y = oracle.rmsnorm(oracle.bf16_to_f64(src[b, h]), wd, w.eps)
            z[b, h] = oracle.rope(y, int(pos[b]), w.rope_theta)
            scale[b, h] = np.abs(y) + np.abs(np.concatenate([y[64:], y[:64]]))
    return z, scale


def check_rounded_rows(got: np.ndarray, want: np.ndarray, z: np.ndarray, window: np.ndarray, what: str) -> int:
    """got/want: bf16 bits of the same rows.  Equal bits, or adjacent values straddling a
    midpoint that the exact value z lies within `window` of.  Returns the tie count."""
    ne = got != want
    if not ne.any():
        return 0
    dist = _midpoint_distance(z[ne], got[ne], want[ne])
    ok = dist <= window[ne]
    assert ok.all(), f"{what}: {int((~ok).sum())} elements differ away from a rounding midpoint"
    return int(ne.sum())


def appended_rows(w: Workload, cache_bits: np.ndarray):
    """The [B, Hkv, d] rows at each sequence's new-token slot of a cache image."""
    rows = cache_bits.reshape(-1, w.Hkv, w.d)
    pos = ints(w.positions)
    out = np.zeros((w.B, w.Hkv, w.d), dtype=np.uint16)
    for b in range(w.B):
        p = int(pos[b])
        if w.paged:
            r = int(ints(w.page_table)[b, p // 64]) * 64 + p % 64
        else:
            r = b * w.max_seq + p
        out[b] = rows[r]
    return out


def rel_l2(a, b) -> float:
    return float(np.linalg.norm(np.asarray(a) - np.asarray(b)) / max(np.linalg.norm(np.asarray(b)), 1e-300))


def ulp_window(x, k: float):
    return k * np.abs(x)


def isclose(a, b):
    return math.isclose(a, b, rel_tol=1e-12)
