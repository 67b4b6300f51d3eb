"""Autoregressive decode: N steps launched back to back on one stream, each attending to the
rows the previous steps appended (seq_len and position advance by one per step, new
q/k/v every step).  Consecutive steps overlap on the device (the next step's attention
kernel starts while the previous step finishes), so this checks that a step reads the
cache only after the previous step's append has landed.  Compared with the fp64 oracle
run step by step on the evolving cache: output per step within the step tolerance, final
caches bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from gqa_decode_attention_fa_gb300 import binding, workloads as wl
from gqa_decode_attention_fa_gb300.workloads import bits, ints

from _util import assert_out_close, geom_of

pytestmark = pytest.mark.gpu

STEPS = 6


def _bf16(gen, shape, device):
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(torch.bfloat16).to(device)


@pytest.mark.parametrize("form,ordered", [(0, False), (-1, False), (16, False), (0, True), (-1, True)])
@pytest.mark.parametrize("paged", [False, True])
def test_back_to_back_autoregressive_steps(paged, form, ordered):
    """form: the planner's choice (the single-launch form here), split-KV + combine, and the
    single-launch form with 16-CTA clusters; ordered: each step's first kernel launched in
    plain stream order (gqa_plan_set_ordered_start)."""
    lens0 = [130, 70, 600]  # no sequence crosses a 64-token page in STEPS steps
    w = wl.make(3, 40, 8, lens0, paged=paged, max_seq=640, seed=41, device="cuda")
    plan = binding.Plan(w.B, w.Hq, w.Hkv, w.max_seq, block_size=w.block_size, num_cache_blocks=w.num_blocks,
                        cluster_size=form)
    if ordered:
        plan.set_ordered_start(True)
    gen = torch.Generator().manual_seed(42)
    steps = []
    for t in range(STEPS):
        sl = torch.tensor([L + t for L in lens0], dtype=torch.int32, device="cuda")
        steps.append(dict(q=_bf16(gen, (w.B, w.Hq, w.d), "cuda"), k=_bf16(gen, (w.B, w.Hkv, w.d), "cuda"),
                          v=_bf16(gen, (w.B, w.Hkv, w.d), "cuda"), sl=sl, pos=sl - 1,
                          out=torch.empty((w.B, w.Hq, w.d), dtype=torch.bfloat16, device="cuda")))
    kc0, vc0 = bits(w.k_cache), bits(w.v_cache)
    for s in steps:  # back to back, no synchronisation in between
        plan.decode_attn(s["q"], s["k"], s["v"], w.k_cache, w.v_cache, w.page_table, s["sl"], s["pos"],
                         w.q_norm_w, w.k_norm_w, w.rope_theta, w.eps, s["out"])
    torch.cuda.synchronize()
    assert plan.device_errors() == 0

    g = geom_of(w)
    kc, vc = kc0, vc0
    for t, s in enumerate(steps):
        ref = oracle.decode_step(g, bits(s["q"]), bits(s["k"]), bits(s["v"]), kc, vc, ints(w.page_table),
                                 ints(s["sl"]), ints(s["pos"]), bits(w.q_norm_w), bits(w.k_norm_w), w.rope_theta,
                                 w.eps)
        assert ref["status"] == 0
        assert_out_close(s["out"], ref["out"], f"step {t}")
        kc, vc = ref["k_cache"], ref["v_cache"]
    np.testing.assert_array_equal(bits(w.v_cache), vc)
    np.testing.assert_array_equal(bits(w.k_cache), kc)


def test_ordered_start_switches_to_the_planners_size_for_a_step_alone():
    """gqa_plan_set_ordered_start re-selects the cluster size: the same as a plan created
    with ordered_start, and back again when cleared; an explicit size is kept."""
    for lens in ([4096], [131072], [256]):
        kw = dict(seq_lens_host=np.asarray(lens, dtype=np.int32))
        overl = binding.Plan(1, 40, 8, max(lens), **kw)
        ordered = binding.Plan(1, 40, 8, max(lens), ordered_start=True, **kw)
        c_overl, c_ordered = overl.cluster_size, ordered.cluster_size
        overl.set_ordered_start(True)
        assert overl.cluster_size == c_ordered
        overl.set_ordered_start(False)
        assert overl.cluster_size == c_overl
        forced = binding.Plan(1, 40, 8, max(lens), cluster_size=2, **kw)
        forced.set_ordered_start(True)
        assert forced.cluster_size == 2
        for p in (overl, ordered, forced):
            p.close()
