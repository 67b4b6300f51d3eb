"""The planner's choices (gqa_plan_describe: no device work) on GB300's description -- 152
SMs; 152 / 76 / 46 / 36 / 28 / 23 / 15 / 15 / 15 / 13 / 8 / 8 / 7 / 7 / 7 / 7 resident
clusters of 1 .. 16 single-launch CTAs (cudaOccupancyMaxActiveClusters on the GPU) --
pinned for the five decode workloads, with overlapping and with ordered step starts, plus
the rules behind them."""
import math

import pytest

from gqa_decode_attention_fa_gb300 import binding, workloads as wl

SMS = binding.GB300_SMS


def describe(w, **kw):
    return binding.plan_describe(w["B"], w["Hq"], w["Hkv"], w["max_seq"], block_size=w.get("block", 0),
                                 num_cache_blocks=w.get("blocks", 0), seq_lens_host=w.get("lens"), **kw)


WORKLOADS = {
    # name: geometry, (split-KV workers, cluster size, splits of the longest segment) with
    # overlapping step starts; the cluster size with ordered starts
    "qwen3-14b-tiny": (dict(B=1, Hq=40, Hkv=8, max_seq=256, lens=[256]), (32, 4, 4), 4),
    "qwen3-14b-4k": (dict(B=1, Hq=40, Hkv=8, max_seq=4096, lens=[4096]), (128, 6, 6), 12),
    "qwen3-14b-ragged": (dict(B=32, Hq=40, Hkv=8, max_seq=8192, block=64, blocks=4000,
                              lens=wl.ragged_lengths(32, 512, 8192, 0)), (152, 1, 1), 1),
    "llama3-70b-128k": (dict(B=1, Hq=64, Hkv=8, max_seq=131072, lens=[131072]), (152, 10, 10), 12),
    "qwen3-14b-40layer": (dict(B=8, Hq=40, Hkv=8, max_seq=32768, block=64, blocks=4096, lens=[32768] * 8),
                          (152, 2, 2), 2),
}


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_choices_on_the_five_workloads(name):
    """Measured on GB300 (graph replay, consecutive steps on different caches, us/step,
    single launch vs split-KV + combine): tiny 4.15 (C=4) vs 6.72; 4k 5.35 (C=6; 5.56 with
    C=10, 5.85 with 8) vs 8.12; ragged 81.6 (C=1) vs 95.1; 128k 75.5 (C=10; 78.6 with 6, 8
    or 12) vs 82.9; one 40-layer layer 145.5 (C=2) vs 163.5.  Each step started in plain
    stream order (no overlap between steps): 4k 8.05 (C=12) vs 9.17 (C=6); 128k 83.1
    (C=12) vs 86.5 (C=10) and 113.4 (C=6)."""
    geom, want, want_ordered = WORKLOADS[name]
    assert describe(geom) == want
    assert describe(geom, ordered_start=True)[1] == want_ordered


def test_split_form_workers_minimise_the_longest_range_then_the_workers():
    """W = ceil(T / ceil(T / SMs)): the longest range is always ceil(T / SMs) tiles (the
    minimum), no worker count below W achieves it, and the rule has no jump where an
    older two-rule fit had one (3 and 4 x SMs)."""
    prev_longest = 0
    for T in list(range(1, 5 * SMS + 2)) + [1000, 5000, 10 ** 5]:
        W, C, _ = binding.plan_describe(1, 8, 1, T * 64, cluster_size=-1)
        assert C == 0 and 1 <= W <= SMS
        longest = math.ceil(T / W)
        assert longest == math.ceil(T / SMS)
        assert W == 1 or math.ceil(T / (W - 1)) > longest
        assert longest >= prev_longest
        prev_longest = longest


def test_cluster_size_rules():
    g = dict(B=1, Hq=40, Hkv=8, max_seq=4096, lens=[4096])
    # 8 segments of 64 tiles: GB300 holds 15 clusters of 7 or 8 CTAs, 23 of 6, so 6 is the
    # largest size with two consecutive steps' 16 clusters resident at once
    assert describe(g)[1] == 6
    # with room for 16 clusters of 9, that size is taken
    roomy = (152, 76, 50, 38, 30, 25, 21, 19, 16, 15, 13, 12, 11, 10, 10, 9)
    assert binding.plan_describe(1, 40, 8, 4096, cluster_capacity=roomy)[1] == 9
    # 64 segments: no size above 1 holds two steps (128 clusters) or one and a half (96);
    # 2 holds one step
    assert binding.plan_describe(8, 40, 8, 32768)[1] == 2
    # long segments (8k: 22 tiles a CTA with clusters of 6, beyond two rings) take the
    # largest size holding one and a half steps (13 clusters of 10 >= 12)
    assert binding.plan_describe(1, 40, 8, 8192)[1] == 10
    # with ordered starts, the largest size holding one step (8 clusters of 12)
    assert binding.plan_describe(1, 40, 8, 8192, ordered_start=True)[1] == 12
    # 40 segments of 64 tiles: no size holds two steps (80 clusters); the segments are long
    # for 2-CTA clusters (32 tiles a CTA), which hold one and a half steps (76 >= 60); with
    # ordered starts 3 (46 >= 40, 120 CTAs)
    assert binding.plan_describe(5, 40, 8, 4096)[1] == 2
    assert binding.plan_describe(5, 40, 8, 4096, ordered_start=True)[1] == 3
    # 16 segments of 64 tiles: 4-CTA clusters hold two steps (36 >= 32) but leave 16 tiles a
    # CTA (long); 5-CTA clusters hold one and a half steps (28 >= 24)
    assert binding.plan_describe(2, 40, 8, 4096)[1] == 5
    # 16 segments of 16 tiles: short, two steps with 4-CTA clusters
    assert binding.plan_describe(2, 40, 8, 1024)[1] == 4
    # a device holding no cluster above 5 CTAs: 5 (40 CTAs, below 48, for 512 tiles) gives
    # way to the split form; with no more tiles than CTAs (5 a segment), to the single launch
    none_above_5 = (152, 76, 46, 36, 28) + (0,) * 11
    assert binding.plan_describe(1, 40, 8, 4096, cluster_capacity=none_above_5)[1] == 0
    assert binding.plan_describe(1, 40, 8, 320, cluster_capacity=none_above_5)[1] == 5
    # never more CTAs per segment than the segment has tiles
    assert binding.plan_describe(1, 40, 8, 100)[1] == 2
    assert binding.plan_describe(1, 40, 8, 64)[1] == 1
    # a long single segment would stream on 16 SMs: split-KV over every SM instead
    assert binding.plan_describe(1, 8, 1, 131072)[1] == 0
    # two long segments on 32 SMs (below 48): split-KV; three on 48 SMs: single launch
    assert binding.plan_describe(1, 16, 2, 131072)[1] == 0
    assert binding.plan_describe(1, 24, 3, 131072)[1] == 16
    # more than two waves of segments: split-KV
    assert binding.plan_describe(64, 40, 8, 1024)[1] == 0
    assert binding.plan_describe(38, 40, 8, 1024)[1] == 1
    # explicit choices
    assert binding.plan_describe(1, 40, 8, 4096, num_workers=64) == (64, 0, 8)
    assert binding.plan_describe(1, 40, 8, 4096, cluster_size=-1)[1] == 0
    assert binding.plan_describe(1, 40, 8, 4096, cluster_size=16)[1] == 16
    assert binding.plan_describe(1, 40, 8, 4096, cluster_size=2)[:2] == (128, 2)


def test_forced_cluster_size_the_device_cannot_hold_is_rejected():
    with pytest.raises(binding.GqaError) as e:
        binding.plan_describe(1, 40, 8, 4096, cluster_size=16,
                              cluster_capacity=binding.GB300_CLUSTER_CAPACITY[:15] + (0,))
    assert e.value.status == binding.GQA_ERR_UNSUPPORTED
    with pytest.raises(binding.GqaError) as e:
        binding.plan_describe(1, 40, 8, 4096, cluster_size=17)
    assert e.value.status == binding.GQA_ERR_INVALID_ARG
    # any size the device holds may be forced, powers of two or not
    assert binding.plan_describe(1, 40, 8, 4096, cluster_size=10)[1] == 10


def test_splits_follow_the_longest_segment():
    # split form: workers whose ranges cover the longest segment (64 tiles over 128 workers' 512)
    assert binding.plan_describe(1, 40, 8, 4096, cluster_size=-1) == (128, 0, 16)
    # single launch: the cluster size (16 segments: 8-CTA clusters would not all fit)
    assert binding.plan_describe(2, 40, 8, 4096, seq_lens_host=[64, 4096]) == (130, 5, 5)
