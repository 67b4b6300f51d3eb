"""GPU parity of the decode step over a 4-bit KV cache (gqa_decode_attn_q4) against the
fp64 oracle.

Output: max |err| <= 1e-2 and relative L2 <= 2e-3, as for the bf16 cache, against the
oracle's attention over the cache the kernel left (so that a near-midpoint index decision,
valid either way, is compared like for like).  Appended rows:
the packed indices equal the oracle's except where the exact rotated coordinate lies within
1e-4 of the midpoint between the two levels (the kernel decides in binary32, the oracle in
binary64), and then the kernel's index is one of those two levels; the scale equals
||z|| / ||c[idx]|| for the kernel's own indices to 1e-5; every other row is untouched.
"""
import dataclasses
import math

import numpy as np
import pytest
import torch

import oracle
from gqa_decode_attention_fa_gb300 import binding, workloads as wl
from gqa_decode_attention_fa_gb300.workloads import bits, ints

from _util import assert_out_close, out_errors

pytestmark = pytest.mark.gpu

D = 128


def np_u8(t):
    return t.detach().contiguous().cpu().numpy()


def oracle_q4(w, pairs=None):
    g = oracle.geom(w.B, w.Hq, w.Hkv, w.d, w.block_size, w.max_seq, w.num_rows)
    return oracle.q4_decode_step(g, bits(w.q_new), bits(w.k_new), bits(w.v_new), np_u8(w.k_idx), np_u8(w.v_idx),
                                 np_u8(w.k_scale), np_u8(w.v_scale), ints(w.page_table), ints(w.seq_lens),
                                 ints(w.positions), bits(w.q_norm_w), bits(w.k_norm_w), w.rope_theta, w.eps,
                                 np_u8(w.rot_signs), bits(w.codebook), pairs=pairs)


def oracle_out_on(w, ref, pairs=None):
    """The oracle's attention over the cache the kernel left (its appended rows checked
    separately), with the oracle's rotated queries."""
    g = oracle.geom(w.B, w.Hq, w.Hkv, w.d, w.block_size, w.max_seq, w.num_rows)
    return oracle.q4_attention(g, ref["q_rot"], np_u8(w.k_idx), np_u8(w.v_idx), np_u8(w.k_scale), np_u8(w.v_scale),
                               ints(w.page_table), ints(w.seq_lens), np_u8(w.rot_signs), bits(w.codebook),
                               pairs=pairs)


# 0: the planner's form (the single-launch form for these small batches), -1: split-KV
FORMS = [0, -1]


def run_gpu(w, cluster_size=0, ordered_start=False):
    plan = binding.Plan(w.B, w.Hq, w.Hkv, w.max_seq, block_size=w.block_size, num_cache_blocks=w.num_blocks,
                        seq_lens_host=w.seq_lens.cpu().numpy(), cluster_size=cluster_size,
                        ordered_start=ordered_start)
    out = torch.full((w.B, w.Hq, w.d), float("nan"), dtype=torch.bfloat16, device="cuda")
    plan.run_q4(w, out)
    torch.cuda.synchronize()
    return plan, out


def new_rows(w):
    pos = ints(w.positions)
    rows = []
    for b in range(w.B):
        p = int(pos[b])
        rows.append(int(ints(w.page_table)[b, p // 64]) * 64 + p % 64 if w.paged else b * w.max_seq + p)
    return rows


def unpack(packed):
    p = packed.astype(np.int64)
    return np.concatenate([p % 16, p // 16])


def check_appended(w, k0, v0, ks0, vs0, ref):
    """Indices as the oracle's up to near-midpoint decisions; scales consistent with the
    kernel's own indices; everything else untouched."""
    c = oracle.bf16_to_f64(bits(w.codebook))
    mid = 0.5 * (c[:-1] + c[1:])
    sg = np_u8(w.rot_signs)
    kw = bits(w.k_norm_w)
    kwd = None if kw is None else oracle.bf16_to_f64(kw)
    ki, vi = np_u8(w.k_idx), np_u8(w.v_idx)
    ks, vs = np_u8(w.k_scale), np_u8(w.v_scale)
    rows = new_rows(w)
    mask = np.ones(ki.shape[0], bool)
    mask[rows] = False
    np.testing.assert_array_equal(ki[mask], k0[mask])
    np.testing.assert_array_equal(vi[mask], v0[mask])
    np.testing.assert_array_equal(ks[mask], ks0[mask])
    np.testing.assert_array_equal(vs[mask], vs0[mask])
    pos = ints(w.positions)
    differing = 0
    for b, r in enumerate(rows):
        for kv in range(w.Hkv):
            for which, got_i, want_i, got_s in (("k", ki, ref["k_idx"], ks), ("v", vi, ref["v_idx"], vs)):
                if which == "k":
                    z = oracle.rope(oracle.rmsnorm(oracle.bf16_to_f64(bits(w.k_new[b, kv])), kwd, w.eps),
                                    int(pos[b]), w.rope_theta)
                else:
                    z = oracle.bf16_to_f64(bits(w.v_new[b, kv]))
                t = math.sqrt(D) * oracle.rotate(z, sg) / np.linalg.norm(z)
                gi, wi = unpack(got_i[r, kv]), unpack(want_i[r, kv])
                for e in np.nonzero(gi != wi)[0]:
                    lo, hi = min(gi[e], wi[e]), max(gi[e], wi[e])
                    assert hi == lo + 1 and abs(t[e] - mid[lo]) < 1e-4, (which, b, kv, e, gi[e], wi[e], t[e])
                    differing += 1
                want_sigma = np.linalg.norm(z) / np.linalg.norm(c[gi])
                assert got_s[r, kv] == pytest.approx(want_sigma, rel=1e-5)
    return differing


CASES = {
    # name: (B, Hq, Hkv, lens, max_seq, paged, qk_norm)
    "g5-contiguous": (2, 40, 8, [130, 600], 640, False, True),
    "g5-paged": (2, 40, 8, [130, 600], 640, True, True),
    "g8-no-norm": (1, 64, 8, [257], 300, False, False),
    "g16-paged": (2, 32, 2, [64, 200], 256, True, True),
    "single-token": (3, 40, 8, [1, 2, 65], 128, True, True),
}


@pytest.mark.parametrize("form", FORMS + [1, 2, 16])
@pytest.mark.parametrize("name", sorted(CASES))
def test_q4_parity(name, form):
    B, Hq, Hkv, lens, max_seq, paged, norm = CASES[name]
    w = wl.make_q4(B, Hq, Hkv, lens, paged=paged, seed=21, qk_norm=norm, max_seq=max_seq, device="cuda", name=name)
    k0, v0, ks0, vs0 = np_u8(w.k_idx), np_u8(w.v_idx), np_u8(w.k_scale), np_u8(w.v_scale)
    ref = oracle_q4(w)
    assert ref["status"] == 0
    plan, out = run_gpu(w, cluster_size=form)
    name = f"{name} [C={plan.cluster_size}]"
    assert plan.device_errors() == 0
    assert check_appended(w, k0, v0, ks0, vs0, ref) <= 2
    want = oracle_out_on(w, ref)
    if name.startswith("single-token"):
        # a one-token context returns its dequantized v row itself, entries up to ~4, where
        # one bf16 rounding alone can exceed 1e-2: allow it per element (2^-7 |ref|)
        got = out.float().cpu().double().numpy()
        assert np.all(np.abs(got - want) <= np.maximum(1e-2, 2.0 ** -7 * np.abs(want)))
        assert out_errors(out, want)[1] <= 2e-3
    else:
        assert_out_close(out, want, name)


def random_q4_geometry(seed):
    """A seeded 4-bit geometry: B in 1..5, H_kv in {1, 2, 4, 8}, G in {1, 2, 3, 5, 7, 16},
    lengths 1..700, paged or contiguous, with or without QK-norm, a capacity that is not a
    tile multiple."""
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 6))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.choice([1, 2, 3, 5, 7, 16]))
    lens = [int(x) for x in rng.integers(1, 701, size=B)]
    return dict(B=B, Hq=G * Hkv, Hkv=Hkv, lens=lens, paged=bool(rng.integers(0, 2)), norm=bool(rng.integers(0, 2)),
                max_seq=max(lens) + int(rng.integers(0, 50)))


@pytest.mark.parametrize("form", FORMS)
@pytest.mark.parametrize("seed", range(5))
def test_q4_random_geometries(seed, form):
    """Five seeded geometries (see random_q4_geometry) in both forms: every output and
    appended row against the oracle."""
    g = random_q4_geometry(3000 + seed)
    w = wl.make_q4(g["B"], g["Hq"], g["Hkv"], g["lens"], paged=g["paged"], seed=seed, qk_norm=g["norm"],
                   max_seq=g["max_seq"], device="cuda", name=f"random-{seed}")
    k0, v0, ks0, vs0 = np_u8(w.k_idx), np_u8(w.v_idx), np_u8(w.k_scale), np_u8(w.v_scale)
    ref = oracle_q4(w)
    assert ref["status"] == 0
    plan, out = run_gpu(w, cluster_size=form)
    assert plan.device_errors() == 0
    assert check_appended(w, k0, v0, ks0, vs0, ref) <= 2
    want = oracle_out_on(w, ref)
    what = f"random geometry {g} [C={plan.cluster_size}]"
    if min(g["lens"]) <= 2:
        # a context of one or two tokens returns (nearly) a dequantized v row, entries up to
        # ~4, where one bf16 rounding can exceed 1e-2: allowed per element (2^-7 |ref|)
        got = out.float().cpu().double().numpy()
        assert np.all(np.abs(got - want) <= np.maximum(1e-2, 2.0 ** -7 * np.abs(want))), what
        assert out_errors(out, want)[1] <= 2e-3, what
    else:
        assert_out_close(out, want, what)


def test_q4_full_size_ragged_on_sampled_heads():
    """The benchmarked ragged batch (32 sequences, 512..8192 tokens, paged): every appended
    row, and 48 sampled (sequence, head) outputs against the oracle."""
    w = wl.named_q4("qwen3-14b-ragged-q4", device="cuda")
    k0, v0, ks0, vs0 = np_u8(w.k_idx), np_u8(w.v_idx), np_u8(w.k_scale), np_u8(w.v_scale)
    pairs = wl.sample_pairs(w.B, w.Hq, 48, seed=22)
    ref = oracle_q4(w, pairs=pairs)
    plan, out = run_gpu(w)
    assert plan.device_errors() == 0
    assert check_appended(w, k0, v0, ks0, vs0, ref) <= 8
    got = torch.stack([out[int(b), int(h)] for b, h in pairs])
    max_abs, rel = out_errors(got, oracle_out_on(w, ref, pairs=pairs))
    assert max_abs <= 1e-2 and rel <= 2e-3, (max_abs, rel)


@pytest.mark.parametrize("ordered", [False, True])
def test_q4_more_segments_than_one_wave(ordered):
    """192 (sequence, KV head) segments of 1..600 tokens -- more one-CTA clusters than the GPU
    holds at once, so that they launch longest first in the plan's order -- with overlapping
    and with ordered starts: every output and appended row against the oracle."""
    lens = wl.ragged_lengths(24, 1, 600, seed=27)
    w = wl.make_q4(24, 16, 8, lens, paged=True, seed=27, max_seq=640, device="cuda", name="one-cta-waves")
    k0, v0, ks0, vs0 = np_u8(w.k_idx), np_u8(w.v_idx), np_u8(w.k_scale), np_u8(w.v_scale)
    ref = oracle_q4(w)
    assert ref["status"] == 0
    plan, out = run_gpu(w, ordered_start=ordered)
    assert plan.cluster_size == 1
    assert plan.device_errors() == 0
    assert check_appended(w, k0, v0, ks0, vs0, ref) <= 8
    assert_out_close(out, oracle_out_on(w, ref), f"one-CTA waves, ordered={ordered}")


@pytest.mark.parametrize("form", FORMS)
def test_q4_plan_reuse_and_determinism(form):
    """Two calls on one plan with the same inputs give the same bits (the second rewrites
    the same rows)."""
    w = wl.make_q4(2, 40, 8, [300, 1000], paged=True, seed=23, max_seq=1024, device="cuda")
    plan, out1 = run_gpu(w, cluster_size=form)
    out2 = torch.empty_like(out1)
    plan.run_q4(w, out2)
    torch.cuda.synchronize()
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


@pytest.mark.parametrize("form", FORMS)
def test_q4_device_index_errors_are_flagged_not_faulted(form):
    """Out-of-range positions, lengths and page ids set error bits and leave the other
    sequences' outputs as they were; a length beyond the capacity zeroes that sequence's
    output; nothing faults (the kernels bound-check; a page outside the pool reads as
    zeros, scales included)."""
    w = wl.make_q4(3, 10, 2, [100, 70, 5], paged=True, seed=24, max_seq=128, device="cuda")
    ref = oracle_q4(w)
    plan, out = run_gpu(w, cluster_size=form)
    assert plan.device_errors() == 0
    want = oracle_out_on(w, ref)
    assert_out_close(out, want, "all valid")
    # position == seq_len for sequence 1
    w.positions[1] = 70
    plan.run_q4(w, out)
    torch.cuda.synchronize()
    assert plan.device_errors() & binding.DEVERR_POSITION
    assert_out_close(out[0:1], want[0:1], "valid sequence beside a bad position")
    # seq_len beyond capacity for sequence 2
    w.positions[1] = 69
    w.seq_lens[2] = w.max_seq + 1
    plan.run_q4(w, out)
    torch.cuda.synchronize()
    assert plan.device_errors() & binding.DEVERR_SEQLEN
    assert torch.count_nonzero(out[2].float()) == 0
    assert_out_close(out[0:1], want[0:1], "valid sequence beside a bad length")
    # page id outside the pool for sequence 1's first page (its new row is on page 1)
    w.seq_lens[2] = 5
    w.page_table[1, 0] = 10 ** 6
    plan.run_q4(w, out)
    torch.cuda.synchronize()
    assert plan.device_errors() & binding.DEVERR_PAGE
    assert plan.device_errors() == 0  # cleared by the previous read
    assert torch.all(torch.isfinite(out.float()))
    assert_out_close(out[0:1], want[0:1], "valid sequence beside a bad page")


@pytest.mark.parametrize("form", FORMS)
def test_q4_back_to_back_steps_match_the_oracle(form):
    """Four autoregressive steps enqueued back to back on one plan and stream, with no host
    synchronisation between them: the lengths grow by one a step and every step brings
    fresh q/k/v.  Each step's output is compared with the oracle's attention over the cache
    the kernels left (later steps append only past this step's length).  Consecutive steps
    overlap on the device, so this checks that no step's kernels run into the previous
    step's reads and that each step sees the rows the previous one appended."""
    base = wl.make_q4(2, 40, 8, [130, 400], paged=True, seed=25, max_seq=448, device="cuda")
    gen = torch.Generator(device="cuda")
    gen.manual_seed(26)
    steps = []
    for s in range(4):  # every input built before the first call
        fresh = [torch.randn(t.shape, generator=gen, device="cuda").to(torch.bfloat16)
                 for t in (base.q_new, base.k_new, base.v_new)]
        steps.append(dataclasses.replace(base, q_new=fresh[0], k_new=fresh[1], v_new=fresh[2],
                                         seq_lens=(base.seq_lens + s).contiguous(),
                                         positions=(base.positions + s).contiguous()))
    plan = binding.Plan(base.B, base.Hq, base.Hkv, base.max_seq, block_size=base.block_size,
                        num_cache_blocks=base.num_blocks, seq_lens_host=base.seq_lens.cpu().numpy(),
                        cluster_size=form)
    outs = [torch.full((base.B, base.Hq, base.d), float("nan"), dtype=torch.bfloat16, device="cuda")
            for _ in steps]
    torch.cuda.synchronize()
    for ws, out in zip(steps, outs):
        plan.run_q4(ws, out)
    torch.cuda.synchronize()
    assert plan.device_errors() == 0
    for s, (ws, out) in enumerate(zip(steps, outs)):
        ref = oracle_q4(ws)
        assert ref["status"] == 0
        assert_out_close(out, oracle_out_on(ws, ref), f"step {s}")
