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

# Rounding acceptance for the appended k rows and the rotated q rows.  A row element is
# RoPE(RMSNorm(x))_i = r (y_i cos - y_partner sin); its computed value differs from the exact
# one by at most WINDOW * (|y_i| + |y_partner|) (double-word k rows: ~2^-44, taken as 2^-40;
# binary32 q rows: norm scalar, cos/sin rounding and one fma, ~2^-20, taken as 2^-18).  An
# element is accepted iff its bf16 value is the round-to-nearest-even of some real within
# that bound of the exact value -- identical bits unless the exact value sits near a rounding
# boundary, or the pair cancels so that the bound spans several bf16 steps.
K_WINDOW = 2.0 ** -40
Q_WINDOW = 2.0 ** -18


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


def _bf16_value(bits_arr: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(bits_arr).view(np.int16)).view(torch.bfloat16).double().numpy()


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


def check_rounded_rows(got: np.ndarray, want: np.ndarray, z: np.ndarray, bound: np.ndarray, what: str) -> int:
    """got/want: bf16 bits of the same rows (library, oracle); z the exact values; bound the
    per-element error bound of the library's arithmetic.  Elements whose bits differ must
    lie in [RNE(z - bound), RNE(z + bound)] (rounding is monotone).  Returns how many
    differ."""
    ne = got != want
    if not ne.any():
        return 0
    zz, bb = z[ne], bound[ne]
    lo = _bf16_value(oracle.round_bf16(zz - bb))
    hi = _bf16_value(oracle.round_bf16(zz + bb))
    g = _bf16_value(got[ne])
    ok = (g >= lo) & (g <= hi)
    if not ok.all():
        idx = np.argwhere(ne)[~ok][:6]
        detail = [(tuple(int(v) for v in i), hex(int(got[tuple(i)])), hex(int(want[tuple(i)])), float(z[tuple(i)]))
                  for i in idx]
        raise AssertionError(f"{what}: {int((~ok).sum())} elements outside the rounding of the exact value "
                             f"+- the error bound: (index, got, want, exact) {detail}")
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
