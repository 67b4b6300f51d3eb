"""gqa_decode_attn_static, the allocation-free entry point: the decode step on the library's
fixed static scratch, compared with gqa_decode_attn (a plan's workspace) on the same inputs
within the step's tolerance (max |err| <= 1e-2, relative L2 <= 2e-3), on consecutive calls.

The file is named to be collected last, so that it also runs after every other GPU test in
one process; it passes on its own in a fresh process as well."""
import numpy as np
import pytest
import torch

from gqa_decode_attention_fa_gb300 import binding, workloads as wl

from _util import MAX_ABS, REL_L2, assert_out_close, oracle_step

pytestmark = pytest.mark.gpu


def _plan_out(w):
    plan = binding.Plan.for_workload(w)
    out = torch.empty((w.B, w.Hq, w.d), dtype=torch.bfloat16, device="cuda")
    plan.run(w, out)
    torch.cuda.synchronize()
    assert plan.device_errors() == 0
    plan.close()
    return out


def _static_out(w, errors):
    out = torch.full((w.B, w.Hq, w.d), float("nan"), dtype=torch.bfloat16, device="cuda")
    binding.decode_attn_static_workload(w, out, device_errors=errors)
    torch.cuda.synchronize()
    return out


def _close(a, b):
    d = (a.float() - b.float()).double()
    max_abs = float(d.abs().max())
    rel = float(torch.linalg.vector_norm(d) / torch.linalg.vector_norm(b.float().double()).clamp_min(1e-300))
    return max_abs <= MAX_ABS and rel <= REL_L2, max_abs, rel


@pytest.mark.parametrize("name", ["qwen3-14b-ragged", "qwen3-14b-4k", "qwen3-14b-tiny"])
def test_static_entry_matches_plan_entry_on_two_calls(name):
    w = wl.named(name, device="cuda")
    ref = _plan_out(w)
    errors = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):
        out = _static_out(w, errors)
        assert torch.isfinite(out.float()).all(), f"call {call}: non-finite output"
        ok, max_abs, rel = _close(out, ref)
        assert ok, f"{name} call {call}: max_abs={max_abs:.3e} rel_l2={rel:.3e} against gqa_decode_attn"
    assert int(errors.item()) == 0


def test_static_entry_alternating_geometries_and_theta():
    """Calls with other batches, cache layouts, group sizes and RoPE bases in between reuse
    the scratch and rebuild the RoPE table when needed; each output still matches the oracle
    and the plan entry."""
    a = wl.make(3, 40, 8, [700, 64, 1], paged=True, seed=21, rope_theta=1e6, device="cuda")
    b = wl.make(2, 64, 4, [3000, 129], paged=False, seed=22, rope_theta=5e5, qk_norm=False, device="cuda")
    c = wl.make(1, 32, 2, [5000], paged=True, seed=23, rope_theta=1e6, max_seq=6000, device="cuda")
    errors = torch.zeros(1, dtype=torch.int32, device="cuda")
    for w in (a, b, a, c, b):
        ref = oracle_step(w)
        out = _static_out(w, errors)
        assert_out_close(out, ref["out"], f"static B={w.B} G={w.Hq // w.Hkv}")
        ok, max_abs, rel = _close(out, _plan_out(w))
        assert ok, f"static vs plan B={w.B}: max_abs={max_abs:.3e} rel_l2={rel:.3e}"
    assert int(errors.item()) == 0


def test_static_entry_back_to_back_calls_with_growing_batch():
    """Calls queued on one stream with no synchronisation between them, the same RoPE base
    and capacity (so the second call reuses the tables and its kernels may start while the
    first call's combine still runs) but a much larger batch, whose rotated-query region in
    the shared scratch covers where the first call's partials lie.  Each output matches the
    oracle."""
    small = wl.make(1, 40, 8, [3000], paged=False, seed=25, max_seq=8192, device="cuda")
    lens = wl.ragged_lengths(32, 512, 8192, seed=26)
    big = wl.make(32, 40, 8, lens, paged=True, seed=26, max_seq=8192, device="cuda")
    refs = [oracle_step(w) for w in (small, big, small)]
    errors = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = [torch.full((w.B, w.Hq, w.d), float("nan"), dtype=torch.bfloat16, device="cuda")
            for w in (small, big, small)]
    # the first call on this geometry builds the tables; then three calls back to back
    binding.decode_attn_static_workload(small, outs[0], device_errors=errors)
    torch.cuda.synchronize()
    for w, out in zip((small, big, small), outs):
        binding.decode_attn_static_workload(w, out, device_errors=errors)
    torch.cuda.synchronize()
    assert int(errors.item()) == 0
    for w, out, ref, tag in zip((small, big, small), outs, refs, ("B=1", "B=32", "B=1 again")):
        assert_out_close(out, ref["out"], f"static back to back {tag}")


def test_static_entry_rejects_geometry_beyond_scratch():
    w = wl.make(1, 8, 2, [100], paged=False, seed=24, device="cuda")
    out = torch.empty((w.B, w.Hq, w.d), dtype=torch.bfloat16, device="cuda")
    # a 131072-token capacity needs 192 MiB of RoPE tables alone (1.5 KiB per position)
    with pytest.raises(binding.GqaError) as e:
        binding.decode_attn_static(1, 8, 2, 131072, w.q_new, w.k_new, w.v_new, w.k_cache, w.v_cache, None,
                                   w.seq_lens, w.positions, w.q_norm_w, w.k_norm_w, w.rope_theta, w.eps, out)
    assert e.value.status == binding.GQA_ERR_SCRATCH_LIMIT
    # argument errors are still reported as such
    with pytest.raises(binding.GqaError) as e:
        binding.decode_attn_static(1, 8, 2, w.max_seq, w.q_new, w.k_new, w.v_new, w.k_cache, w.v_cache, None,
                                   w.seq_lens, w.positions, w.q_norm_w, w.k_norm_w, -1.0, w.eps, out)
    assert e.value.status == binding.GQA_ERR_INVALID_ARG
    # and the scratch still serves a valid call afterwards
    ref = oracle_step(w)
    errors = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert_out_close(_static_out(w, errors), ref["out"], "static after rejected calls")
    assert np.all(int(errors.item()) == 0)
