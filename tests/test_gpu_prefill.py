"""GPU parity of the chunked causal prefill (gqa_prefill_attn) against the fp64 oracle.

Output: max |err| <= 1e-2 and relative L2 <= 2e-3 over the call's whole output (the same
acceptance as the decode step).  Cache: the chunk's k rows bit-exact (the double-word
computation may differ only within 2^-40 (|y_i| + |y_partner|) of a bf16 rounding
boundary), its v rows bit copies, every other row untouched.  Cases cover G = 1, 3, 5, 8
and 16 (query blocks of 128, 42, 25, 16 and 8 tokens, the last one ragged), paged and
contiguous caches, chunks at the prompt start and deep into it, one-token chunks, a prompt
fed in several chunks, out-of-range chunks, and the full-size workload on sampled rows.
"""
import numpy as np
import pytest
import torch

import oracle
from gqa_decode_attention_fa_gb300 import binding, workloads as wl
from gqa_decode_attention_fa_gb300.workloads import bits, ints

from _util import K_WINDOW, assert_out_close, check_rounded_rows, out_errors

pytestmark = pytest.mark.gpu

DEV = binding.DEVERR_POSITION | binding.DEVERR_SEQLEN | binding.DEVERR_PAGE | binding.DEVERR_TIMEOUT


def geom(w):
    return oracle.geom(w.B, w.Hq, w.Hkv, w.d, w.block_size, w.max_seq, w.num_rows)


def oracle_prefill(w, triples=None):
    return oracle.prefill_step(geom(w), w.T, bits(w.q_new), bits(w.k_new), bits(w.v_new), bits(w.k_cache),
                               bits(w.v_cache), ints(w.page_table), ints(w.q_start), bits(w.q_norm_w),
                               bits(w.k_norm_w), w.rope_theta, w.eps, triples=triples)


def run_gpu(w, err=None):
    out = torch.full((w.B, w.T, w.Hq, w.d), float("nan"), dtype=torch.bfloat16, device="cuda")
    binding.prefill_attn_workload(w, out, device_errors=err)
    torch.cuda.synchronize()
    return out


def cache_row(w, b, t):
    if w.paged:
        return int(ints(w.page_table)[b, t // 64]) * 64 + t % 64
    return b * w.max_seq + t


def exact_k_rows(w, b, i):
    """Exact fp64 RMSNorm + RoPE of chunk token i's k rows, and the per-element slack scale."""
    kw = bits(w.k_norm_w)
    wd = None if kw is None else oracle.bf16_to_f64(kw)
    p = int(ints(w.q_start)[b]) + i
    src = bits(w.k_new[b, i])
    z = np.zeros((w.Hkv, w.d))
    sc = np.zeros((w.Hkv, w.d))
    for kv in range(w.Hkv):
        y = oracle.rmsnorm(oracle.bf16_to_f64(src[kv]), wd, w.eps)
        z[kv] = oracle.rope(y, p, w.rope_theta)
        sc[kv] = np.abs(y) + np.abs(np.concatenate([y[64:], y[:64]]))
    return z, sc


def check_cache(w, k0, v0, ref, seqs=None):
    """Appended rows as the oracle's (k within the rounding window, v bit copies), the rest
    of both caches untouched."""
    kc = bits(w.k_cache).reshape(-1, w.Hkv, w.d)
    vc = bits(w.v_cache).reshape(-1, w.Hkv, w.d)
    k0, v0 = k0.reshape(kc.shape), v0.reshape(vc.shape)
    rk, rv = ref["k_cache"].reshape(kc.shape), ref["v_cache"].reshape(vc.shape)
    np.testing.assert_array_equal(vc, rv)
    mask = np.ones(kc.shape[0], bool)
    starts = ints(w.q_start)
    for b in (range(w.B) if seqs is None else seqs):
        for i in range(w.T):
            r = cache_row(w, b, int(starts[b]) + i)
            mask[r] = False
            if not np.array_equal(kc[r], rk[r]):
                z, sc = exact_k_rows(w, b, i)
                check_rounded_rows(kc[r], rk[r], z, K_WINDOW * sc, f"k row (b={b}, i={i})")
    np.testing.assert_array_equal(kc[mask], k0[mask])
    np.testing.assert_array_equal(vc[mask], v0[mask])


CASES = {
    # name: (B, Hq, Hkv, T, starts, max_seq, paged, qk_norm, theta)
    "g5-contiguous": (2, 40, 8, 77, [0, 130], 256, False, True, 1e6),
    "g5-paged": (2, 40, 8, 77, [0, 130], 256, True, True, 1e6),
    "g8-no-norm": (1, 64, 8, 100, [200], 320, False, False, 5e5),
    "g1-paged": (1, 8, 8, 150, [37], 192, True, True, 1e6),
    "g16-paged": (1, 32, 2, 40, [64], 128, True, True, 1e6),
    "g3-contiguous": (3, 12, 4, 50, [0, 5, 90], 160, False, True, 1e6),
    "one-token-chunks": (3, 40, 8, 1, [0, 63, 200], 256, True, True, 1e6),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_prefill_parity(name):
    B, Hq, Hkv, T, starts, max_seq, paged, norm, theta = CASES[name]
    w = wl.make_prefill(B, Hq, Hkv, T, starts, paged=paged, seed=11, qk_norm=norm, rope_theta=theta,
                        max_seq=max_seq, device="cuda", name=name)
    k0, v0 = bits(w.k_cache), bits(w.v_cache)
    ref = oracle_prefill(w)
    assert ref["status"] == 0
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run_gpu(w, err)
    assert int(err.item()) == 0
    assert_out_close(out, ref["out"], name)
    check_cache(w, k0, v0, ref)


def random_geometry(seed):
    """A seeded prefill geometry: B in 1..3, H_kv in {1, 2, 4, 8}, G in {1, 2, 3, 4, 6, 7, 12}
    (query blocks of 128, 64, 42, 32, 21, 18 and 10 tokens), T in 1..200, chunk starts
    anywhere (not tile-aligned), paged or contiguous, with or without QK-norm."""
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 4))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.choice([1, 2, 3, 4, 6, 7, 12]))
    T = int(rng.integers(1, 201))
    max_seq = int(rng.integers(T, T + 320))
    starts = [int(x) for x in rng.integers(0, max_seq - T + 1, size=B)]
    return dict(B=B, Hq=G * Hkv, Hkv=Hkv, T=T, starts=starts, max_seq=max_seq, paged=bool(rng.integers(0, 2)),
                norm=bool(rng.integers(0, 2)))


@pytest.mark.parametrize("seed", range(8))
def test_random_geometries(seed):
    """Eight seeded geometries (see random_geometry): every output row and appended row
    against the oracle, and no device error."""
    g = random_geometry(1000 + seed)
    w = wl.make_prefill(g["B"], g["Hq"], g["Hkv"], g["T"], g["starts"], paged=g["paged"], seed=seed,
                        qk_norm=g["norm"], max_seq=g["max_seq"], device="cuda", name=f"random-{seed}")
    k0, v0 = bits(w.k_cache), bits(w.v_cache)
    ref = oracle_prefill(w)
    assert ref["status"] == 0
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run_gpu(w, err)
    assert int(err.item()) == 0, g
    assert_out_close(out, ref["out"], f"random geometry {g}")
    check_cache(w, k0, v0, ref)


def test_v_values_far_from_unit_scale():
    """P V keeps V's bf16 range: KV head 2's values scaled by 2^-20 (every value far below
    fp16's normal range), KV head 5 holding 70000 in a cache row and -1e6 in a chunk row
    (beyond fp16's largest), the other heads ordinary.  Every KV head but 5 is held to the
    relative L2 bound on its own scale; head 5's outputs, up to ~10^4, element by element to
    one bf16 step of the exact value plus 10^-3 of the head's largest."""
    B, Hq, Hkv, T = 1, 40, 8, 77
    w = wl.make_prefill(B, Hq, Hkv, T, [130], paged=False, seed=5, max_seq=256, device="cuda", name="v-range")
    w.v_cache[:, :, 2] *= 2.0 ** -20
    w.v_new[:, :, 2] *= 2.0 ** -20
    w.v_cache[0, 10, 5, 7] = 70000.0
    w.v_new[0, 40, 5, 100] = -1e6
    ref = oracle_prefill(w)
    assert ref["status"] == 0
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run_gpu(w, err)
    assert int(err.item()) == 0
    g = out.float().cpu().double().numpy().reshape(T, Hkv, Hq // Hkv, w.d)
    r = ref["out"].reshape(T, Hkv, Hq // Hkv, w.d)
    assert np.all(np.isfinite(g))
    rels = {kv: float(np.linalg.norm(g[:, kv] - r[:, kv]) / np.linalg.norm(r[:, kv])) for kv in range(Hkv) if kv != 5}
    assert max(rels.values()) <= 2e-3, rels
    big = np.abs(r[:, 5])
    assert np.all(np.abs(g[:, 5] - r[:, 5]) <= 2.0 ** -8 * big + 1e-3 * big.max())


def test_prompt_fed_in_chunks_matches_one_call():
    """A 300-token prompt through three calls (128 + 128 + 44 tokens, each on the cache the
    previous one left) gives the outputs of the oracle's single 300-token chunk."""
    w = wl.make_prefill(1, 40, 8, 300, [0], paged=True, seed=12, max_seq=320, device="cuda")
    ref = oracle_prefill(w)
    outs = []
    for a, e in ((0, 128), (128, 256), (256, 300)):
        part = wl.PrefillWorkload(**{**w.__dict__, "T": e - a, "q_new": w.q_new[:, a:e].contiguous(),
                                     "k_new": w.k_new[:, a:e].contiguous(), "v_new": w.v_new[:, a:e].contiguous(),
                                     "q_start": torch.tensor([a], dtype=torch.int32, device="cuda")})
        outs.append(run_gpu(part))
    assert_out_close(torch.cat(outs, dim=1), ref["out"], "chunked prompt")
    np.testing.assert_array_equal(bits(w.v_cache), ref["v_cache"])


def test_repeated_calls_are_bitwise_identical():
    """The kernels are deterministic: a race between the pipeline roles (a read of the
    accumulator before its last product landed, a tile overwritten early) would show as
    run-to-run differences.  Twelve calls of a 512-token chunk, then twelve of a chunked
    prompt whose query blocks see one to five KV tiles."""
    w = wl.make_prefill(1, 40, 8, 512, [1536], paged=False, seed=16, max_seq=2048, device="cuda")
    first = run_gpu(w)
    for _ in range(11):
        assert torch.equal(run_gpu(w).view(torch.int16), first.view(torch.int16))
    w = wl.make_prefill(1, 40, 8, 300, [0], paged=True, seed=12, max_seq=320, device="cuda")
    k0, v0 = w.k_cache.clone(), w.v_cache.clone()
    runs = []
    for _ in range(12):
        w.k_cache.copy_(k0)
        w.v_cache.copy_(v0)
        outs = []
        for a, e in ((0, 128), (128, 256), (256, 300)):
            part = wl.PrefillWorkload(**{**w.__dict__, "T": e - a, "q_new": w.q_new[:, a:e].contiguous(),
                                         "k_new": w.k_new[:, a:e].contiguous(), "v_new": w.v_new[:, a:e].contiguous(),
                                         "q_start": torch.tensor([a], dtype=torch.int32, device="cuda")})
            outs.append(run_gpu(part))
        runs.append(torch.cat(outs, dim=1).view(torch.int16))
    for r in runs[1:]:
        assert torch.equal(r, runs[0])


CHUNKS_300 = ((0, 128), (128, 256), (256, 300))


def chunk_parts(w):
    """The 300-token prompt's three calls: each chunk's q/k/v in tensors of its own."""
    return [wl.PrefillWorkload(**{**w.__dict__, "T": e - a, "q_new": w.q_new[:, a:e].contiguous(),
                                  "k_new": w.k_new[:, a:e].contiguous(), "v_new": w.v_new[:, a:e].contiguous(),
                                  "q_start": torch.tensor([a], dtype=torch.int32, device="cuda")})
            for a, e in CHUNKS_300]


def test_calls_queued_back_to_back_and_replayed_from_a_graph():
    """Each call's attention kernel reads what its own prologue wrote, and each call's
    prologue waits for the previous call's readers of `out` and the cache.  The 300-token
    prompt's three calls queued on one stream with no synchronisation between them; then the
    same three calls captured in a CUDA graph and replayed on two other prompts (fresh
    inputs and cache copied in before each replay), every output against the oracle's."""
    w = wl.make_prefill(1, 40, 8, 300, [0], paged=True, seed=21, max_seq=320, device="cuda")
    k0, v0 = w.k_cache.clone(), w.v_cache.clone()
    ref = oracle_prefill(w)
    parts = chunk_parts(w)
    outs = [torch.full((1, e - a, 40, 128), float("nan"), dtype=torch.bfloat16, device="cuda") for a, e in CHUNKS_300]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for part, out in zip(parts, outs):
        binding.prefill_attn_workload(part, out, device_errors=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_out_close(torch.cat(outs, dim=1), ref["out"], "queued calls")

    w.k_cache.copy_(k0)
    w.v_cache.copy_(v0)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for part, out in zip(parts, outs):
            binding.prefill_attn_workload(part, out, device_errors=err, stream=s)
    for seed in (22, 23):
        w2 = wl.make_prefill(1, 40, 8, 300, [0], paged=True, seed=seed, max_seq=320, device="cuda")
        ref2 = oracle_prefill(w2)
        for name in ("k_cache", "v_cache", "page_table", "q_norm_w", "k_norm_w"):
            getattr(w, name).copy_(getattr(w2, name))
        for (a, e), part in zip(CHUNKS_300, parts):
            part.q_new.copy_(w2.q_new[:, a:e])
            part.k_new.copy_(w2.k_new[:, a:e])
            part.v_new.copy_(w2.v_new[:, a:e])
        for out in outs:
            out.fill_(float("nan"))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_out_close(torch.cat(outs, dim=1), ref2["out"], f"graph replay, prompt {seed}")


def test_out_of_range_chunks_give_zeros_and_flags():
    """Sequence 1's chunk runs past max_seq_len and sequence 2's starts before 0: both are
    flagged, write no cache row and output zeros; sequence 0 is unaffected."""
    w = wl.make_prefill(3, 40, 8, 20, [10, 250, 0], paged=False, seed=13, max_seq=256, device="cuda")
    w.q_start[2] = -3
    k0, v0 = bits(w.k_cache), bits(w.v_cache)
    w_ok = wl.PrefillWorkload(**{**w.__dict__, "B": 1, "q_new": w.q_new[:1], "k_new": w.k_new[:1],
                                 "v_new": w.v_new[:1], "k_cache": w.k_cache[:1].clone(),
                                 "v_cache": w.v_cache[:1].clone(), "q_start": w.q_start[:1]})
    ref0 = oracle_prefill(w_ok)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run_gpu(w, err)
    e = int(err.item())
    assert e & binding.DEVERR_SEQLEN and e & binding.DEVERR_POSITION and not e & binding.DEVERR_TIMEOUT
    assert_out_close(out[:1], ref0["out"], "valid sequence")
    assert torch.count_nonzero(out[1:]).item() == 0
    kc = bits(w.k_cache)
    np.testing.assert_array_equal(kc[1:], k0[1:])
    np.testing.assert_array_equal(bits(w.v_cache)[1:], v0[1:])


def test_rejects_bad_arguments():
    w = wl.make_prefill(1, 40, 8, 8, [0], paged=False, seed=14, max_seq=64, device="cuda")
    out = torch.empty((1, 8, 40, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(binding.GqaError) as ex:   # a page table for a contiguous cache
        binding.prefill_attn(1, 40, 8, 8, 64, w.q_new, w.k_new, w.v_new, w.k_cache, w.v_cache,
                             torch.zeros((1, 1), dtype=torch.int32, device="cuda"), w.q_start, w.q_norm_w,
                             w.k_norm_w, 1e6, 1e-6, out)
    assert ex.value.status == binding.GQA_ERR_INVALID_ARG
    with pytest.raises(binding.GqaError) as ex:   # chunk longer than the capacity
        binding.prefill_attn(1, 40, 8, 65, 64, w.q_new, w.k_new, w.v_new, w.k_cache, w.v_cache, None, w.q_start,
                             w.q_norm_w, w.k_norm_w, 1e6, 1e-6, out)
    assert ex.value.status == binding.GQA_ERR_INVALID_ARG
    with pytest.raises(binding.GqaError) as ex:   # misaligned output
        flat = torch.empty(1 * 8 * 40 * 128 + 8, dtype=torch.bfloat16, device="cuda")
        binding.prefill_attn(1, 40, 8, 8, 64, w.q_new, w.k_new, w.v_new, w.k_cache, w.v_cache, None, w.q_start,
                             w.q_norm_w, w.k_norm_w, 1e6, 1e-6, flat[1:1 + 8 * 40 * 128])
    assert ex.value.status == binding.GQA_ERR_INVALID_ARG


def test_two_sequences_with_tiles_cut_into_kv_parts():
    """Two sequences of a 640-token chunk (416 query tiles of 25 tokens x 5 heads on a
    152-SM GPU: 304 whole tiles, the last 112 cut into KV parts merged by the third
    kernel), paged, at different cache offsets: every output row and appended row against
    the oracle."""
    w = wl.make_prefill(2, 40, 8, 640, [0, 200], paged=True, seed=16, max_seq=896, device="cuda", name="cut-b2")
    k0, v0 = bits(w.k_cache), bits(w.v_cache)
    ref = oracle_prefill(w)
    assert ref["status"] == 0
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run_gpu(w, err)
    assert int(err.item()) == 0
    assert_out_close(out, ref["out"], "two sequences, cut tiles")
    check_cache(w, k0, v0, ref)


def test_full_size_workload_on_sampled_rows():
    """The benchmarked chunk (1024 tokens at positions 3072..4095 over a 4096-token cache):
    every appended k/v row against the oracle's prologue, and the output on 96 sampled
    (token, head) rows -- the first and last tokens, both sides of every query-block edge
    near the start, and random ones -- against the oracle's attention over the oracle's
    cache."""
    w = wl.named_prefill("qwen3-14b-prefill-4k", device="cuda")
    g = geom(w)
    q_rot, kc_ref, vc_ref, st = oracle.prefill_prologue(
        g, w.T, bits(w.q_new), bits(w.k_new), bits(w.v_new), bits(w.k_cache), bits(w.v_cache), None,
        ints(w.q_start), bits(w.q_norm_w), bits(w.k_norm_w), w.rope_theta, w.eps)
    assert st == 0
    k0, v0 = bits(w.k_cache), bits(w.v_cache)
    out = run_gpu(w)
    check_cache(w, k0, v0, dict(k_cache=kc_ref, v_cache=vc_ref))
    rng = np.random.default_rng(15)
    toks = sorted(set([0, 1, 24, 25, 26, 49, 50, 511, 512, 1000, 1022, 1023] +
                      [int(x) for x in rng.choice(w.T, 36, replace=False)]))
    triples = [(0, int(t), int(h)) for t in toks for h in rng.choice(w.Hq, 2, replace=False)]
    ref, _ = oracle.prefill_attention(g, w.T, q_rot, kc_ref, vc_ref, None, ints(w.q_start), triples=triples)
    got = torch.stack([out[b, t, h] for b, t, h in triples])
    max_abs, rel = out_errors(got, ref)
    assert torch.isfinite(out.float()).all()
    assert max_abs <= 1e-2 and rel <= 2e-3, (max_abs, rel)
