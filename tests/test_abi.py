"""CPU checks of the C ABI: the library loads and exports every function the header
declares, host-side validation rejects bad geometry before touching a device, and the
split-KV partition covers every tile exactly once in contiguous, balanced ranges."""
import ctypes

import numpy as np
import pytest

from gqa_decode_attention_fa_gb300 import binding


def test_library_exports_every_declared_function():
    lib = binding.load()
    names = binding.header_functions()
    assert "gqa_decode_attn" in names and "gqa_plan_create" in names
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings():
    lib = binding.load()
    for s in range(5):
        assert lib.gqa_status_string(s)
    assert binding.status_string(1) == "invalid argument"


def _create(**over):
    d = dict(batch=2, num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=64, max_seq_len=128,
             num_cache_blocks=4, num_workers=0, device=0, cluster_size=0, ordered_start=0)
    d.update(over)
    desc = binding.PlanDesc(*[d[n] for n, _ in binding.PlanDesc._fields_])
    h = ctypes.c_void_p()
    return binding.load().gqa_plan_create(ctypes.byref(desc), None, ctypes.byref(h))


@pytest.mark.parametrize("over,status", [
    (dict(batch=0), binding.GQA_ERR_INVALID_ARG),
    (dict(num_q_heads=0), binding.GQA_ERR_INVALID_ARG),
    (dict(max_seq_len=0), binding.GQA_ERR_INVALID_ARG),
    (dict(num_workers=-1), binding.GQA_ERR_INVALID_ARG),
    (dict(block_size=-64), binding.GQA_ERR_INVALID_ARG),
    (dict(num_cache_blocks=0), binding.GQA_ERR_INVALID_ARG),
    (dict(cluster_size=17), binding.GQA_ERR_INVALID_ARG),
    (dict(cluster_size=32), binding.GQA_ERR_INVALID_ARG),
    (dict(cluster_size=-2), binding.GQA_ERR_INVALID_ARG),
    (dict(head_dim=64), binding.GQA_ERR_UNSUPPORTED),
    (dict(num_q_heads=10, num_kv_heads=4), binding.GQA_ERR_UNSUPPORTED),   # H_q % H_kv != 0
    (dict(num_q_heads=34, num_kv_heads=2), binding.GQA_ERR_UNSUPPORTED),   # G = 17
    (dict(batch=1025), binding.GQA_ERR_UNSUPPORTED),
    (dict(block_size=32), binding.GQA_ERR_UNSUPPORTED),
    (dict(block_size=0, batch=1024, max_seq_len=1 << 21), binding.GQA_ERR_UNSUPPORTED),  # rows > 2^31
])
def test_plan_create_rejects_bad_geometry(over, status):
    assert _create(**over) == status


def test_null_arguments_are_rejected():
    lib = binding.load()
    assert lib.gqa_plan_create(None, None, None) == binding.GQA_ERR_INVALID_ARG
    args = [None] * 11 + [ctypes.c_float(1e6), ctypes.c_float(1e-6), None, None]
    assert lib.gqa_decode_attn(*args) == binding.GQA_ERR_INVALID_ARG
    assert lib.gqa_decode_attn_host(*args) == binding.GQA_ERR_INVALID_ARG
    f1, f2 = ctypes.c_float(1e6), ctypes.c_float(1e-6)
    assert lib.gqa_attention_splitkv(None, None, None, None, None, None, None, None, None, None, None, f1, f2,
                                     None) == binding.GQA_ERR_INVALID_ARG
    assert lib.gqa_combine(None, None, None, None) == binding.GQA_ERR_INVALID_ARG
    assert lib.gqa_plan_destroy(None) == binding.GQA_OK
    assert lib.gqa_plan_num_workers(None) == 0
    assert lib.gqa_plan_num_splits(None) == 0
    assert lib.gqa_plan_set_ordered_start(None, 1) == binding.GQA_ERR_INVALID_ARG
    assert lib.gqa_plan_cluster_size(None) == 0
    f = ctypes.c_uint32()
    assert lib.gqa_plan_device_errors(None, ctypes.byref(f), 0) == binding.GQA_ERR_INVALID_ARG


@pytest.mark.parametrize("lens,hkv,W", [
    ([256], 8, 32), ([4096], 8, 152), ([131072], 8, 152), ([1, 64, 65, 1000], 2, 7),
    ([1, 64, 65, 1000], 2, 1000), ([5, 0, 7], 3, 4),
])
def test_partition_covers_every_tile_once_in_balanced_contiguous_ranges(lens, hkv, W):
    max_seq = max(max(lens), 1)
    T, rng = binding.partition_describe(lens, hkv, max_seq, W)
    tiles = [(L + 63) // 64 if 1 <= L <= max_seq else 0 for L in lens]
    assert T == hkv * sum(tiles)
    assert rng[0, 0] == 0 and rng[-1, 1] == T
    assert np.all(rng[1:, 0] == rng[:-1, 1])                 # contiguous, no gaps or overlaps
    sizes = rng[:, 1] - rng[:, 0]
    assert sizes.min() >= 0 and sizes.max() - sizes.min() <= 1  # balanced to one tile


def test_partition_worker_lookup_agrees_with_ranges():
    """The kernels find a tile's worker arithmetically as floor(((x+1)W - 1)/T); check it
    against the published ranges for many (T, W)."""
    for T in (1, 2, 31, 32, 33, 1000, 16384, 17411):
        for W in (1, 2, 3, 7, 152, 1000):
            _, rng = binding.partition_describe([64 * T], 1, 64 * T, W)
            for x in set([0, T - 1, T // 2, T // 3] + list(range(0, T, max(1, T // 50)))):
                w = ((x + 1) * W - 1) // T
                assert rng[w, 0] <= x < rng[w, 1]


# ----------------------------------------------------------------------------- prefill entry

def _prefill(**over):
    """gqa_prefill_attn with non-null dummy tensors: rejected on its arguments before any
    device work (the pointers are never dereferenced)."""
    d = dict(batch=1, num_q_heads=40, num_kv_heads=8, head_dim=128, chunk_len=16, block_size=0,
             max_seq_len=64, num_cache_blocks=0, device=0)
    d.update(over)
    desc = binding.PrefillDesc(*[d[n] for n, _ in binding.PrefillDesc._fields_])
    dummy = ctypes.c_void_p(4096)
    pt = dummy if d["block_size"] else None
    return binding.load().gqa_prefill_attn(ctypes.byref(desc), dummy, dummy, dummy, dummy, dummy, pt, dummy, None,
                                           None, ctypes.c_float(1e6), ctypes.c_float(1e-6), dummy, None, None)


@pytest.mark.parametrize("over,status", [
    (dict(batch=0), binding.GQA_ERR_INVALID_ARG),
    (dict(chunk_len=0), binding.GQA_ERR_INVALID_ARG),
    (dict(chunk_len=65), binding.GQA_ERR_INVALID_ARG),          # longer than the capacity
    (dict(head_dim=64), binding.GQA_ERR_UNSUPPORTED),
    (dict(num_q_heads=34, num_kv_heads=2), binding.GQA_ERR_UNSUPPORTED),   # G = 17
    (dict(num_q_heads=10, num_kv_heads=4), binding.GQA_ERR_UNSUPPORTED),   # H_q % H_kv != 0
    (dict(block_size=32), binding.GQA_ERR_UNSUPPORTED),
    (dict(block_size=64, num_cache_blocks=0), binding.GQA_ERR_INVALID_ARG),
    (dict(batch=1025), binding.GQA_ERR_INVALID_ARG),
])
def test_prefill_rejects_bad_geometry(over, status):
    assert _prefill(**over) == status


def test_prefill_rejects_null_and_inconsistent_arguments():
    lib = binding.load()
    args = [None] * 10 + [ctypes.c_float(1e6), ctypes.c_float(1e-6), None, None, None]
    assert lib.gqa_prefill_attn(*args) == binding.GQA_ERR_INVALID_ARG      # NULL desc
    desc = binding.PrefillDesc(1, 40, 8, 128, 16, 0, 64, 0, 0)
    dummy = ctypes.c_void_p(4096)
    # a page table for a contiguous cache
    assert lib.gqa_prefill_attn(ctypes.byref(desc), dummy, dummy, dummy, dummy, dummy, dummy, dummy, None, None,
                                ctypes.c_float(1e6), ctypes.c_float(1e-6), dummy, None, None) == binding.GQA_ERR_INVALID_ARG
    # theta <= 0
    assert lib.gqa_prefill_attn(ctypes.byref(desc), dummy, dummy, dummy, dummy, dummy, None, dummy, None, None,
                                ctypes.c_float(0.0), ctypes.c_float(1e-6), dummy, None, None) == binding.GQA_ERR_INVALID_ARG
    # a misaligned bf16 tensor
    odd = ctypes.c_void_p(4096 + 2)
    assert lib.gqa_prefill_attn(ctypes.byref(desc), odd, dummy, dummy, dummy, dummy, None, dummy, None, None,
                                ctypes.c_float(1e6), ctypes.c_float(1e-6), dummy, None, None) == binding.GQA_ERR_INVALID_ARG


# ----------------------------------------------------------------------------- 4-bit cache entry

def test_q4_codebook_is_the_lloyd_max_quantizer():
    """The library's levels (its own Lloyd iteration) round to the oracle's, level by level."""
    import oracle
    import torch
    want = torch.tensor(oracle.lloyd_max(16)[0], dtype=torch.float32).to(torch.bfloat16)
    np.testing.assert_array_equal(binding.q4_codebook(), want.view(torch.int16).numpy().view(np.uint16))
    assert binding.load().gqa_q4_codebook(None) == binding.GQA_ERR_INVALID_ARG


def test_q4_rejects_null_arguments():
    args = [None] * 15 + [ctypes.c_float(1e6), ctypes.c_float(1e-6), None, None]
    assert binding.load().gqa_decode_attn_q4(*args) == binding.GQA_ERR_INVALID_ARG
