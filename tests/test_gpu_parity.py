"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the same seeded
inputs.  Output: max |err| <= 1e-2 and relative L2 <= 2e-3.  Appended cache rows: bit-exact
(the double-word computation may differ only within 2^-40 (|y_i| + |y_partner|) of a bf16
rounding boundary; no such element is expected), every other cache row untouched; rotated
q: the bf16 rounding of a value within the binary32 error bound of the exact value."""
import numpy as np
import pytest
import torch

import oracle
from gqa_decode_attention_fa_gb300 import binding, workloads as wl
from gqa_decode_attention_fa_gb300.workloads import bits, ints

from _util import (K_WINDOW, Q_WINDOW, appended_rows, assert_out_close, check_rounded_rows, oracle_step,
                   rotated_rows)

pytestmark = pytest.mark.gpu


# The step's two forms: 0 lets the planner choose (the single-launch form for the small
# batches most tests use), -1 forces split-KV + combine.
FORMS = [0, -1]


def run_gpu(w, plan=None, num_workers=0, cluster_size=0, ordered_start=False):
    plan = plan or binding.Plan.for_workload(w, num_workers=num_workers, cluster_size=cluster_size)
    if ordered_start:
        plan.set_ordered_start(True)
    out = torch.empty((w.B, w.Hq, w.d), dtype=torch.bfloat16, device="cuda")
    plan.run(w, out)
    torch.cuda.synchronize()
    return plan, out


def full_check(w, num_workers=0, what="", cluster_size=0, ordered_start=False):
    """Run both sides on workload w (on the GPU) and check output, cache and q."""
    k0, v0 = bits(w.k_cache), bits(w.v_cache)
    ref = oracle_step(w)
    assert ref["status"] == 0
    plan, out = run_gpu(w, num_workers=num_workers, cluster_size=cluster_size, ordered_start=ordered_start)
    what = f"{what} [C={plan.cluster_size}]"
    assert plan.device_errors() == 0
    stats = assert_out_close(out, ref["out"], what)
    # cache: only the appended rows may change, V bit copies, K bit-exact (midpoint ties aside)
    kc, vc = bits(w.k_cache), bits(w.v_cache)
    np.testing.assert_array_equal(vc, ref["v_cache"])
    rows_g, rows_o = appended_rows(w, kc), appended_rows(w, ref["k_cache"])
    mask = np.ones(kc.reshape(-1, w.Hkv, w.d).shape[0], bool)
    pos = ints(w.positions)
    for b in range(w.B):
        p = int(pos[b])
        r = int(ints(w.page_table)[b, p // 64]) * 64 + p % 64 if w.paged else b * w.max_seq + p
        mask[r] = False
    np.testing.assert_array_equal(kc.reshape(-1, w.Hkv, w.d)[mask], k0.reshape(-1, w.Hkv, w.d)[mask])
    zk, sk = rotated_rows(w, "k")
    diff_k = check_rounded_rows(rows_g, rows_o, zk, K_WINDOW * sk, f"{what} k rows")
    assert diff_k == 0   # double-word arithmetic: bit-exact in practice
    zq, sq = rotated_rows(w, "q")
    diff_q = check_rounded_rows(plan.read_q_rot(), ref["q_rot"], zq, Q_WINDOW * sq, f"{what} q rows")
    assert diff_q <= max(4, zq.size // 1000)
    del k0, v0
    return stats, plan, out


# ------------------------------------------------------------------ the named workloads

@pytest.mark.parametrize("name", ["qwen3-14b-tiny", "qwen3-14b-4k", "qwen3-14b-ragged", "llama3-70b-128k"])
def test_named_workload_full_parity(name):
    w = wl.named(name, device="cuda")
    full_check(w, what=name)


@pytest.mark.parametrize("name", ["qwen3-14b-4k", "qwen3-14b-ragged"])
def test_named_workloads_with_ordered_starts(name):
    """Ordered starts re-select the cluster size (12 on the 4k step) and, for the ragged
    batch (more one-CTA clusters than SMs), launch its segments longest first."""
    w = wl.named(name, device="cuda")
    full_check(w, what=f"{name} ordered", ordered_start=True)


@pytest.mark.parametrize("name", ["qwen3-14b-tiny", "qwen3-14b-4k"])
def test_named_short_workloads_in_the_split_form(name):
    """The planner runs these in the single-launch form; the split-KV form must agree too."""
    w = wl.named(name, device="cuda")
    full_check(w, what=name, cluster_size=-1)


@pytest.mark.parametrize("csize", [1, 2, 3, 4, 8, 10, 16])
@pytest.mark.parametrize("Hq,Hkv,lens,paged", [
    (40, 8, [1000, 1, 64, 65], True),     # G = 5, ragged, single-token and page-edge lengths
    (64, 8, [4096], False),               # G = 8
    (32, 2, [700, 129], True),            # G = 16 (two head blocks)
    (8, 8, [300, 2000], False),           # G = 1
])
def test_single_launch_cluster_sizes(csize, Hq, Hkv, lens, paged):
    """Cluster sizes of the single-launch form, forced, including sizes that do not divide
    the 128 dims (uneven dim slices), sizes larger than a short sequence's tile count (CTAs
    with no tiles) and non-portable 16-CTA clusters."""
    w = wl.make(len(lens), Hq, Hkv, lens, paged=paged, seed=csize * 100 + Hq + len(lens), device="cuda")
    full_check(w, what=f"C={csize} G={Hq // Hkv} lens={lens}", cluster_size=csize)


def test_40_layer_sweep_parity():
    """All 40 layers of the sweep through one plan, as the benchmark runs them: three layers
    checked in full, every layer checked on all heads of one sampled sequence."""
    plan = None
    out = None
    rng = np.random.default_rng(0)
    for layer in range(wl.LAYERS_40):
        w = wl.named("qwen3-14b-40layer", device="cuda", layer=layer)
        if plan is None:
            plan = binding.Plan.for_workload(w)
            out = torch.empty((w.B, w.Hq, w.d), dtype=torch.bfloat16, device="cuda")
        if layer in (0, 17, 39):
            full_check(w, what=f"layer {layer}")
            del w
            torch.cuda.empty_cache()
            continue
        b = int(rng.integers(0, w.B))
        plan.run(w, out)
        torch.cuda.synchronize()
        # one sequence, gathered to a contiguous single-sequence problem for the oracle
        k, v = wl.gather_sequence(w, b)
        L = int(w.seq_lens[b].item())
        g = oracle.geom(1, w.Hq, w.Hkv, w.d, 0, k.shape[0], k.shape[0])
        pos = ints(w.positions)[b:b + 1]
        # the caches were already updated by the library: the oracle re-runs the prologue
        # on the same new-token inputs, which rewrites the same slot with its own values
        ref = oracle.decode_step(g, bits(w.q_new[b:b + 1]), bits(w.k_new[b:b + 1]), bits(w.v_new[b:b + 1]),
                                 bits(k), bits(v), None, np.array([L], np.int32), pos, bits(w.q_norm_w),
                                 bits(w.k_norm_w), w.rope_theta, w.eps)
        assert ref["status"] == 0
        assert_out_close(out[b:b + 1], ref["out"], f"layer {layer} seq {b}")
        del w, k, v
    assert plan.device_errors() == 0


# ------------------------------------------------------------------ edge cases

@pytest.mark.parametrize("form", FORMS)
@pytest.mark.parametrize("lens", [[1], [2], [63], [64], [65], [127, 128, 129], [1, 64, 65, 300, 7]])
@pytest.mark.parametrize("paged", [False, True])
def test_ragged_tails_and_tiny_lengths(lens, paged, form):
    w = wl.make(len(lens), 10, 2, lens, paged=paged, seed=len(lens) * 7 + 1, device="cuda", extra_blocks=3)
    full_check(w, what=f"lens={lens} paged={paged}", cluster_size=form)


@pytest.mark.parametrize("form", FORMS)
@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (4, 2), (8, 2), (10, 2), (16, 2), (24, 2), (32, 2), (64, 8)])
def test_group_sizes(Hq, Hkv, form):
    w = wl.make(3, Hq, Hkv, [70, 200, 5], paged=True, seed=Hq + Hkv, device="cuda")
    full_check(w, what=f"G={Hq // Hkv}", cluster_size=form)


@pytest.mark.parametrize("qk_norm", [False, True])
def test_with_and_without_qk_norm(qk_norm):
    w = wl.make(2, 40, 8, [300, 1000], paged=False, qk_norm=qk_norm, seed=3, device="cuda")
    full_check(w, what=f"qk_norm={qk_norm}")


def test_one_sided_norm_weights():
    w = wl.make(2, 8, 2, [100, 33], paged=True, seed=4, device="cuda")
    w.k_norm_w = None
    full_check(w, what="q norm only")
    w = wl.make(2, 8, 2, [100, 33], paged=True, seed=5, device="cuda")
    w.q_norm_w = None
    full_check(w, what="k norm only")


@pytest.mark.parametrize("form", FORMS)
def test_new_token_mid_sequence_and_capacity_not_a_tile_multiple(form):
    w = wl.make(3, 10, 2, [100, 150, 37], paged=False, max_seq=150, positions=[10, 149, 0], seed=6,
                device="cuda")
    full_check(w, what="positions < L-1, max_seq=150", cluster_size=form)


def random_decode_geometry(seed):
    """A seeded decode geometry: B in 1..6, H_kv in {1, 2, 4, 8}, G in {1, 2, 3, 5, 6, 7, 16},
    lengths 1..700 (positions L_b - 1, or anywhere below L_b for some sequences), paged
    or contiguous, with or without QK-norm, and a capacity that is not a tile multiple."""
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 7))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.choice([1, 2, 3, 5, 6, 7, 16]))
    lens = [int(x) for x in rng.integers(1, 701, size=B)]
    positions = [int(rng.integers(0, L)) if rng.integers(0, 3) == 0 else L - 1 for L in lens]
    return dict(B=B, Hq=G * Hkv, Hkv=Hkv, lens=lens, positions=positions, paged=bool(rng.integers(0, 2)),
                norm=bool(rng.integers(0, 2)), max_seq=max(lens) + int(rng.integers(0, 50)))


@pytest.mark.parametrize("form", FORMS)
@pytest.mark.parametrize("seed", range(6))
def test_random_geometries(seed, form):
    """Six seeded geometries (see random_decode_geometry) in both forms: output, cache and
    rotated queries against the oracle."""
    g = random_decode_geometry(2000 + seed)
    w = wl.make(g["B"], g["Hq"], g["Hkv"], g["lens"], paged=g["paged"], seed=seed, qk_norm=g["norm"],
                positions=g["positions"], max_seq=g["max_seq"], device="cuda", name=f"random-{seed}")
    full_check(w, what=f"random geometry {g} form {form}", cluster_size=form)


@pytest.mark.parametrize("workers", [1, 2, 3, 7, 64, 151, 1000])
def test_worker_counts(workers):
    w = wl.make(5, 40, 8, [1, 700, 64, 3000, 129], paged=True, seed=8, device="cuda")
    full_check(w, num_workers=workers, what=f"W={workers}")


def test_large_scores_and_outliers_are_stable():
    """K outliers x20 (as in the 40-layer sweep) and a long context on a small batch."""
    w = wl.make(2, 40, 8, [20000, 9000], paged=True, seed=9, k_outlier_frac=0.01, device="cuda")
    full_check(w, what="outliers")


@pytest.mark.parametrize("Hq,Hkv", [(40, 8), (24, 2)])
def test_many_short_segments_per_worker(Hq, Hkv):
    """Short sequences put many (sequence, KV head) segments into one worker's range, so
    the query-rotation ring wraps (G <= 8 and G > 8 layouts)."""
    rng = np.random.default_rng(15)
    lens = rng.integers(1, 200, size=96).tolist()
    w = wl.make(96, Hq, Hkv, lens, paged=True, seed=16, device="cuda")
    full_check(w, what=f"short segments G={Hq // Hkv}")
    full_check(w, num_workers=7, what=f"short segments G={Hq // Hkv} W=7")


def test_max_batch():
    lens = (np.arange(1024) % 97 + 1).tolist()
    w = wl.make(1024, 8, 2, lens, paged=True, seed=10, device="cuda")
    full_check(w, what="B=1024")


# ------------------------------------------------------------------ API behaviour

def test_plans_of_different_batches_coexist():
    """A plan made after another one, for a smaller batch, leaves the first one usable (the
    attention kernel's shared-memory limit is set for the largest batch, not per plan)."""
    big = wl.make(256, 8, 2, (np.arange(256) % 97 + 1).tolist(), paged=True, seed=13, device="cuda")
    small = wl.make(1, 8, 2, [100], paged=False, seed=14, device="cuda")
    ref = oracle_step(big)
    plan_big = binding.Plan.for_workload(big)
    plan_small = binding.Plan.for_workload(small)
    out = torch.empty((big.B, big.Hq, big.d), dtype=torch.bfloat16, device="cuda")
    plan_big.run(big, out)
    torch.cuda.synchronize()
    assert plan_big.device_errors() == 0
    assert_out_close(out, ref["out"], "B=256 after a B=1 plan")
    run_gpu(small, plan=plan_small)


def test_plan_reused_across_changed_lengths():
    """One plan, calls whose lengths (and so the tile partition) change: the first tiles
    each worker prefetches from the previous call's partition are then wrong guesses, which
    must cost nothing but time."""
    w1 = wl.make(2, 40, 8, [3000, 1000], paged=False, max_seq=4096, seed=31, device="cuda")
    w2 = wl.make(2, 40, 8, [1500, 4000], paged=False, max_seq=4096, seed=32, device="cuda")
    plan = binding.Plan(2, 40, 8, 4096)
    for w in (w1, w2, w1):
        ref = oracle_step(w)
        out = torch.empty((w.B, w.Hq, w.d), dtype=torch.bfloat16, device="cuda")
        plan.run(w, out)
        torch.cuda.synchronize()
        assert plan.device_errors() == 0
        assert_out_close(out, ref["out"], f"lengths {ints(w.seq_lens).tolist()}")


@pytest.mark.parametrize("form", FORMS)
def test_step_replays_from_a_cuda_graph(form):
    """After a first eager call (which builds the RoPE tables) the step can be captured into
    a CUDA graph; replays give the eager output bit for bit."""
    w = wl.make(4, 40, 8, [500, 64, 1, 2000], paged=True, seed=15, device="cuda")
    plan, out_eager = run_gpu(w, cluster_size=form)
    out = torch.empty_like(out_eager)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        plan.run(w, out, s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        plan.run(w, out, s)
    for _ in range(2):
        out.zero_()
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), out_eager.view(torch.int16))
    assert plan.device_errors() == 0


@pytest.mark.parametrize("name", ["qwen3-14b-ragged", "qwen3-14b-4k"])
def test_determinism_bitwise(name):
    w = wl.named(name, device="cuda")
    plan, out1 = run_gpu(w)
    out2 = torch.empty_like(out1)
    plan.run(w, out2)
    torch.cuda.synchronize()
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


def test_steps_equal_fused_call():
    """In the split-KV form, the step's two launch entry points in order give the fused
    call's output bit for bit."""
    w = wl.make(4, 40, 8, [500, 64, 1, 2000], paged=True, seed=11, device="cuda")
    plan, out1 = run_gpu(w, cluster_size=-1)
    assert plan.cluster_size == 0
    out2 = torch.empty_like(out1)
    plan.run_steps(w, out2)
    torch.cuda.synchronize()
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


@pytest.mark.parametrize("pinned", [True, False])
def test_host_buffer_entry_point_matches_device_call(pinned):
    """Page-locked host buffers are read and written in place by the kernels; pageable ones
    go through the staging copies.  Both give the device entry point's output bit for bit."""
    w = wl.make(4, 40, 8, [500, 64, 1, 2000], paged=True, seed=12, device="cuda")
    plan, out1 = run_gpu(w)
    pin = (lambda t: t.pin_memory()) if pinned else (lambda t: t)
    host = {k: pin(getattr(w, k).cpu()) for k in ("q_new", "k_new", "v_new", "seq_lens", "positions")}
    out_h = pin(torch.empty((w.B, w.Hq, w.d), dtype=torch.bfloat16))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        plan.decode_attn_host(host["q_new"], host["k_new"], host["v_new"], w.k_cache, w.v_cache, w.page_table,
                              host["seq_lens"], host["positions"], w.q_norm_w, w.k_norm_w, w.rope_theta, w.eps,
                              out_h, stream=s)
    s.synchronize()
    assert torch.equal(out1.cpu().view(torch.int16), out_h.view(torch.int16))


@pytest.mark.parametrize("form", FORMS)
def test_device_index_errors_are_flagged_not_faulted(form):
    """Out-of-range positions, lengths and page ids set error bits, zero that sequence's
    output and leave the others correct; nothing faults (the kernels bound-check)."""
    w = wl.make(3, 10, 2, [100, 70, 5], paged=True, seed=13, device="cuda", extra_blocks=2)
    ref = oracle_step(w)
    plan = binding.Plan.for_workload(w, cluster_size=form)
    out = torch.empty((w.B, w.Hq, w.d), dtype=torch.bfloat16, device="cuda")
    # position == seq_len for sequence 1
    w.positions[1] = 70
    plan.run(w, out)
    assert plan.device_errors() & binding.DEVERR_POSITION
    # seq_len beyond capacity for sequence 2
    w.positions[1] = 69
    w.seq_lens[2] = w.max_seq + 1
    plan.run(w, out)
    assert plan.device_errors() & binding.DEVERR_SEQLEN
    assert torch.count_nonzero(out[2].float()) == 0
    assert_out_close(out[0:1], ref["out"][0:1], "valid sequence beside a bad one")
    # page id outside the pool for sequence 0's first page
    w.seq_lens[2] = 5
    w.page_table[0, 0] = 10 ** 6
    plan.run(w, out)
    assert plan.device_errors() & binding.DEVERR_PAGE
    assert plan.device_errors() == 0  # cleared by the previous read


def test_host_validation_rejects_bad_arguments():
    w = wl.make(2, 8, 2, [10, 20], paged=True, seed=14, device="cuda")
    plan = binding.Plan.for_workload(w)
    out = torch.empty((w.B, w.Hq, w.d), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(binding.GqaError) as e:
        plan.decode_attn(w.q_new, w.k_new, w.v_new, w.k_cache, w.v_cache, None, w.seq_lens, w.positions,
                         w.q_norm_w, w.k_norm_w, w.rope_theta, w.eps, out)
    assert e.value.status == binding.GQA_ERR_INVALID_ARG
    with pytest.raises(binding.GqaError) as e:
        plan.decode_attn(w.q_new, w.k_new, w.v_new, w.k_cache, w.v_cache, w.page_table, w.seq_lens, w.positions,
                         w.q_norm_w, w.k_norm_w, -1.0, w.eps, out)
    assert e.value.status == binding.GQA_ERR_INVALID_ARG
    with pytest.raises(binding.GqaError) as e:
        plan.decode_attn(w.q_new, w.k_new, w.v_new, w.k_cache, w.v_cache, w.page_table, w.seq_lens, w.positions,
                         w.q_norm_w, w.k_norm_w, w.rope_theta, float("nan"), out)
    assert e.value.status == binding.GQA_ERR_INVALID_ARG
    # misaligned device tensors are rejected before anything is launched
    q_shift = torch.empty(w.q_new.numel() + 1, dtype=torch.bfloat16, device="cuda")[1:].view_as(w.q_new)
    q_shift.copy_(w.q_new)
    with pytest.raises(binding.GqaError) as e:
        plan.decode_attn(q_shift, w.k_new, w.v_new, w.k_cache, w.v_cache, w.page_table, w.seq_lens, w.positions,
                         w.q_norm_w, w.k_norm_w, w.rope_theta, w.eps, out)
    assert e.value.status == binding.GQA_ERR_INVALID_ARG
    out_shift = torch.empty(out.numel() + 4, dtype=torch.bfloat16, device="cuda")[4:].view_as(out)
    with pytest.raises(binding.GqaError) as e:
        plan.decode_attn(w.q_new, w.k_new, w.v_new, w.k_cache, w.v_cache, w.page_table, w.seq_lens, w.positions,
                         w.q_norm_w, w.k_norm_w, w.rope_theta, w.eps, out_shift)
    assert e.value.status == binding.GQA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    with pytest.raises(binding.GqaError) as e:
        binding.Plan(2, 8, 2, 64, block_size=64, num_cache_blocks=0)
    assert e.value.status == binding.GQA_ERR_INVALID_ARG
    with pytest.raises(binding.GqaError) as e:
        binding.Plan(2, 8, 2, 64, head_dim=64)
    assert e.value.status == binding.GQA_ERR_UNSUPPORTED
    with pytest.raises(binding.GqaError) as e:
        binding.Plan(2, 34, 2, 64)
    assert e.value.status == binding.GQA_ERR_UNSUPPORTED
