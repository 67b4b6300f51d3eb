"""Pins of the chunked-prefill oracle (CPU only).

The prefill oracle states causal attention of a block of T new tokens over the cache
("ADR-0060: AHBM GQA Fused Attention Kernel (Llama3-70B)", section 5.4).  Each test ties
it to something other than itself: the already-pinned decode step (a chunk of one token
is one decode step), closed forms (equal scores give the running mean of V over the
visible prefix; one visible key gives its V row), causality (no output moves when a later
token changes), independence of how the prompt is cut into chunks, and the page's own
past / partial / future tile classes, which must give the brute-force result.  A slip in
the causal bound (< instead of <=), the query-head -> KV-head map, the chunk offset or
the token index of a row fails one of them.
"""
import numpy as np
import pytest
import torch

import oracle

D = 128


def bf(x):
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def f64(bits):
    return torch.from_numpy(np.asarray(bits, dtype=np.uint16).view(np.int16)).view(torch.bfloat16).double().numpy()


def make_case(B, Hq, Hkv, T, q_start, max_seq, paged, seed, norm=True):
    """Random chunk inputs and a filled cache (rows past each sequence's q_start are
    filled too: the prologue must overwrite the chunk's rows and attention must not read
    past the query's position)."""
    rng = np.random.default_rng(seed)
    if paged:
        bs = 64
        max_blocks = (max_seq + bs - 1) // bs
        nblk = B * max_blocks
        perm = rng.permutation(nblk).astype(np.int32)
        pt = perm.reshape(B, max_blocks)
        rows = nblk * bs
    else:
        bs, pt, rows = 0, None, B * max_seq
    g = oracle.geom(B, Hq, Hkv, D, bs, max_seq, rows)
    c = dict(
        g=g, T=T,
        q_new=bf(rng.standard_normal((B, T, Hq, D))),
        k_new=bf(rng.standard_normal((B, T, Hkv, D))),
        v_new=bf(rng.standard_normal((B, T, Hkv, D))),
        k_cache=bf(rng.standard_normal((rows, Hkv, D))),
        v_cache=bf(rng.standard_normal((rows, Hkv, D))),
        page_table=pt,
        q_start=np.asarray(q_start, dtype=np.int32),
        q_norm_w=bf(1.0 + 0.1 * rng.standard_normal(D)) if norm else None,
        k_norm_w=bf(1.0 + 0.1 * rng.standard_normal(D)) if norm else None,
        rope_theta=1e6, eps=1e-6,
    )
    return c


def run(c, **kw):
    args = {k: c[k] for k in ("q_new", "k_new", "v_new", "k_cache", "v_cache", "page_table", "q_start",
                              "q_norm_w", "k_norm_w", "rope_theta", "eps")}
    args.update(kw)
    return oracle.prefill_step(c["g"], c["T"], **args)


def cache_row(c, b, t):
    g = c["g"]
    if c["page_table"] is None:
        return b * g.max_seq + t
    return int(c["page_table"][b, t // 64]) * 64 + t % 64


# ----------------------------------------------------------------------------- one token

@pytest.mark.parametrize("paged", [False, True])
def test_chunk_of_one_token_is_a_decode_step(paged):
    """T = 1 at q_start = s is exactly the decode step with seq_len s + 1, position s:
    same rotated q, same cache rows, bit-identical output (the decode oracle is pinned
    independently to closed forms in test_oracle_pins.py)."""
    c = make_case(3, 8, 2, 1, [0, 63, 130], 192, paged, seed=1)
    r = run(c)
    assert r["status"] == 0
    d = oracle.decode_step(c["g"], c["q_new"][:, 0], c["k_new"][:, 0], c["v_new"][:, 0], c["k_cache"],
                           c["v_cache"], c["page_table"], c["q_start"] + 1, c["q_start"], c["q_norm_w"],
                           c["k_norm_w"], c["rope_theta"], c["eps"])
    assert d["status"] == 0
    np.testing.assert_array_equal(r["q_rot"][:, 0], d["q_rot"])
    np.testing.assert_array_equal(r["k_cache"], d["k_cache"])
    np.testing.assert_array_equal(r["v_cache"], d["v_cache"])
    np.testing.assert_array_equal(r["out"][:, 0], d["out"])


def test_every_chunk_row_is_the_decode_prologue_at_its_position():
    """Token i of the chunk is rotated at position q_start + i and lands in that slot."""
    c = make_case(2, 4, 2, 9, [5, 60], 128, True, seed=2)
    r = run(c)
    g = c["g"]
    for b in range(2):
        for i in range(c["T"]):
            p = int(c["q_start"][b]) + i
            gb = oracle.geom(1, g.Hq, g.Hkv, D, g.block_size, g.max_seq, g.num_rows)
            pt = None if c["page_table"] is None else c["page_table"][b:b + 1]
            q_rot, kc, vc, st = oracle.prologue(gb, c["q_new"][b, i][None], c["k_new"][b, i][None],
                                                c["v_new"][b, i][None], c["k_cache"], c["v_cache"], pt,
                                                np.array([p + 1], np.int32), np.array([p], np.int32),
                                                c["q_norm_w"], c["k_norm_w"], c["rope_theta"], c["eps"])
            assert st == 0
            np.testing.assert_array_equal(r["q_rot"][b, i], q_rot[0])
            row = cache_row(c, b, p)
            np.testing.assert_array_equal(r["k_cache"][row], kc[row])
            np.testing.assert_array_equal(r["v_cache"][row], c["v_new"][b, i])


# ----------------------------------------------------------------------------- closed forms

@pytest.mark.parametrize("paged", [False, True])
def test_equal_scores_give_the_mean_of_the_visible_prefix(paged):
    """q = 0 makes every score 0, so token i's output is the plain mean of V_t over
    t = 0 .. q_start + i (inclusive: the token sees itself), with the chunk's own v rows
    in place of whatever the cache held at those slots."""
    c = make_case(2, 6, 3, 21, [0, 77], 192, paged, seed=3)
    c["q_new"] = np.zeros_like(c["q_new"])
    r = run(c)
    assert r["status"] == 0
    g = c["g"]
    G = g.Hq // g.Hkv
    for b in range(2):
        s = int(c["q_start"][b])
        for kv in range(g.Hkv):
            rows = [f64(c["v_cache"][cache_row(c, b, t), kv]) for t in range(s)]
            rows += [f64(c["v_new"][b, i, kv]) for i in range(c["T"])]
            V = np.stack(rows)
            prefix_mean = np.cumsum(V, axis=0) / np.arange(1, len(V) + 1)[:, None]
            for i in range(c["T"]):
                for h in range(kv * G, kv * G + G):
                    np.testing.assert_allclose(r["out"][b, i, h], prefix_mean[s + i], rtol=0, atol=1e-12)


def test_first_prompt_token_returns_its_own_v():
    """At q_start = 0 the first token sees one key, itself: out = its v row exactly."""
    c = make_case(2, 8, 4, 5, [0, 0], 64, False, seed=4)
    r = run(c)
    G = 2
    for b in range(2):
        for h in range(8):
            np.testing.assert_array_equal(r["out"][b, 0, h], f64(c["v_new"][b, 0, h // G]))


def test_query_head_reads_its_own_kv_head():
    """V constant per KV head (c_kv everywhere) makes out[., ., h] = c_{floor(h/G)}: a wrong
    head map or a wrong G fails."""
    c = make_case(1, 6, 3, 7, [40], 64, False, seed=5)
    consts = np.array([0.5, -2.0, 3.0])
    c["v_cache"] = np.broadcast_to(bf(consts)[None, :, None], c["v_cache"].shape).copy()
    c["v_new"] = np.broadcast_to(bf(consts)[None, None, :, None], c["v_new"].shape).copy()
    r = run(c)
    for h in range(6):
        np.testing.assert_allclose(r["out"][0, :, h], consts[h // 2], rtol=0, atol=1e-14)


# ----------------------------------------------------------------------------- invariants

def test_causality_later_tokens_do_not_move_earlier_outputs():
    c = make_case(1, 4, 2, 12, [30], 64, False, seed=6)
    base = run(c)
    j = 7
    c2 = dict(c)
    c2["k_new"] = c["k_new"].copy()
    c2["v_new"] = c["v_new"].copy()
    c2["k_new"][:, j:] = bf(np.random.default_rng(60).standard_normal(c["k_new"][:, j:].shape))
    c2["v_new"][:, j:] = bf(np.random.default_rng(61).standard_normal(c["v_new"][:, j:].shape))
    moved = run(c2)
    np.testing.assert_array_equal(moved["out"][:, :j], base["out"][:, :j])
    assert np.all(np.abs(moved["out"][:, j] - base["out"][:, j]).max(axis=-1) > 1e-6)


def test_cache_rows_past_the_chunk_are_never_read():
    """The cache past q_start + T holds garbage (here: huge values); it must not matter."""
    c = make_case(1, 4, 2, 10, [20], 128, False, seed=7)
    base = run(c)
    c2 = dict(c)
    c2["k_cache"] = c["k_cache"].copy()
    c2["v_cache"] = c["v_cache"].copy()
    c2["k_cache"][30:] = bf(np.full(c["k_cache"][30:].shape, 1e30))
    c2["v_cache"][30:] = bf(np.full(c["v_cache"][30:].shape, -1e30))
    np.testing.assert_array_equal(run(c2)["out"], base["out"])


@pytest.mark.parametrize("paged", [False, True])
def test_chunking_does_not_change_the_result(paged):
    """One chunk of 20 tokens == a chunk of 8 followed by a chunk of 12 on the updated cache."""
    c = make_case(2, 4, 2, 20, [3, 64], 128, paged, seed=8)
    whole = run(c)
    a = dict(c, T=8, q_new=c["q_new"][:, :8], k_new=c["k_new"][:, :8], v_new=c["v_new"][:, :8])
    ra = run(a)
    bpart = dict(c, T=12, q_new=c["q_new"][:, 8:], k_new=c["k_new"][:, 8:], v_new=c["v_new"][:, 8:],
                 k_cache=ra["k_cache"], v_cache=ra["v_cache"], q_start=c["q_start"] + 8)
    rb = run(bpart)
    np.testing.assert_array_equal(np.concatenate([ra["out"], rb["out"]], axis=1), whole["out"])
    np.testing.assert_array_equal(rb["k_cache"], whole["k_cache"])
    np.testing.assert_array_equal(rb["v_cache"], whole["v_cache"])


@pytest.mark.parametrize("q_block,kv_tile", [(1, 1), (5, 7), (16, 64), (64, 16), (37, 128), (128, 64)])
def test_tile_classes_match_brute_force(q_block, kv_tile):
    """The past / partial (triangular mask) / future (skipped) classes of the page's
    prefill kernel, run as online softmax, equal the plain definition."""
    c = make_case(2, 4, 2, 37, [0, 50], 128, True, seed=9)
    r = run(c)
    g = c["g"]
    for b in range(2):
        for h in (0, 3):
            got = oracle.prefill_blocked(g, c["T"], r["q_rot"], r["k_cache"], r["v_cache"], c["page_table"],
                                         c["q_start"], b, h, q_block, kv_tile)
            np.testing.assert_allclose(got, r["out"][b, :, h], rtol=0, atol=1e-12)


def test_sampled_triples_match_the_full_output():
    c = make_case(2, 4, 2, 9, [10, 3], 64, False, seed=10)
    r = run(c)
    tr = [(0, 0, 0), (1, 8, 3), (0, 4, 2), (1, 0, 1)]
    got, _ = oracle.prefill_attention(c["g"], c["T"], r["q_rot"], r["k_cache"], r["v_cache"], None,
                                      c["q_start"], triples=tr)
    for k, (b, i, h) in enumerate(tr):
        np.testing.assert_array_equal(got[k], r["out"][b, i, h])


# ----------------------------------------------------------------------------- errors

def test_out_of_range_chunks_are_reported_and_not_written():
    c = make_case(2, 4, 2, 10, [60, -1], 64, False, seed=11)
    r = run(c)
    assert r["status"] in (1, 2)
    np.testing.assert_array_equal(r["k_cache"], c["k_cache"])
    c = make_case(1, 4, 2, 10, [55], 64, False, seed=11)
    assert run(c)["status"] == 2
    c = make_case(1, 4, 2, 10, [54], 64, False, seed=11)
    assert run(c)["status"] == 0
