"""Seeded synthetic inputs for the decode step.

This module only draws random tensors; it holds none of the step's arithmetic.  Both the
CUDA path and the fp64 oracle consume exactly the tensors built here (the oracle as raw
bf16 bits), so nothing else is shared between them.

Draw recipe (fixed order per workload): lengths, q/k/v of the new token, QK-norm weights,
K cache, V cache, K outliers, page-table permutation.  Normal draws are fp32 and rounded to
bf16 by ``Tensor.to(torch.bfloat16)`` (round to nearest even).

Named workloads (the five decode geometries the step is measured on):

* ``qwen3-14b-tiny``    B=1, 40/8 heads, d=128, L=256 (new token at 255), contiguous cache,
  QK-norm weights ~N(1, 0.1), eps 1e-6, theta 1e6.
* ``qwen3-14b-4k``      B=1, 40/8, L=4096, contiguous, QK-norm, theta 1e6.
* ``qwen3-14b-ragged``  B=32, 40/8, L_b ~ U{512..8192}, paged (64-token blocks, randomly
  permuted page table), QK-norm, theta 1e6.
* ``llama3-70b-128k``   B=1, 64/8 (G=8), L=131072, contiguous, no QK-norm, theta 5e5.
* ``qwen3-14b-40layer`` 40 layers x (B=8, 40/8, L=32768, paged, per-layer page tables,
  1 % of K-cache elements scaled x20 before rounding), QK-norm, theta 1e6.

And one sweep over steps (``decode_sweep``): ``qwen3-14b-4k-decode``, 64 autoregressive
steps through 40 layers of the 4k geometry, the length growing from 4033 to 4096.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np
import torch

HEAD_DIM = 128
BLOCK = 64


@dataclasses.dataclass
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    block_size: int          # 64 = paged, 0 = contiguous
    max_seq: int             # per-sequence capacity
    num_blocks: int          # paged pool size in blocks (0 when contiguous)
    rope_theta: float
    eps: float
    q_new: torch.Tensor      # [B, Hq, d] bf16
    k_new: torch.Tensor      # [B, Hkv, d] bf16
    v_new: torch.Tensor      # [B, Hkv, d] bf16
    k_cache: torch.Tensor    # paged [nb, 64, Hkv, d] or contiguous [B, max_seq, Hkv, d] bf16
    v_cache: torch.Tensor
    page_table: Optional[torch.Tensor]  # [B, ceil(max_seq/64)] int32, -1 where unused
    seq_lens: torch.Tensor   # [B] int32
    positions: torch.Tensor  # [B] int32
    q_norm_w: Optional[torch.Tensor]    # [d] bf16
    k_norm_w: Optional[torch.Tensor]

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def paged(self) -> bool:
        return self.block_size > 0

    @property
    def max_blocks(self) -> int:
        return -(-self.max_seq // BLOCK)

    @property
    def num_rows(self) -> int:
        return self.num_blocks * BLOCK if self.paged else self.B * self.max_seq

    def kv_bytes(self) -> int:
        """Bytes of K and V the step must read: sum_b L_b * H_kv * d * 2 tensors * 2 B."""
        return int(self.seq_lens.long().sum().item()) * self.Hkv * self.d * 2 * 2

    def to(self, device) -> "Workload":
        def mv(t):
            return None if t is None else t.to(device)
        return dataclasses.replace(
            self, q_new=mv(self.q_new), k_new=mv(self.k_new), v_new=mv(self.v_new),
            k_cache=mv(self.k_cache), v_cache=mv(self.v_cache), page_table=mv(self.page_table),
            seq_lens=mv(self.seq_lens), positions=mv(self.positions),
            q_norm_w=mv(self.q_norm_w), k_norm_w=mv(self.k_norm_w))


def bits(t: Optional[torch.Tensor]) -> Optional[np.ndarray]:
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    if t is None:
        return None
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def ints(t: Optional[torch.Tensor]) -> Optional[np.ndarray]:
    if t is None:
        return None
    return t.detach().contiguous().cpu().numpy().astype(np.int32)


def _normal_bf16(gen: torch.Generator, shape, device, scale: float = 1.0, mean: float = 0.0):
    x = torch.randn(shape, generator=gen, dtype=torch.float32, device=device)
    if scale != 1.0:
        x.mul_(scale)
    if mean != 0.0:
        x.add_(mean)
    return x.to(torch.bfloat16)


def make(B: int, Hq: int, Hkv: int, lens: Sequence[int], *, paged: bool, seed: int = 0,
         qk_norm: bool = True, rope_theta: float = 1e6, eps: float = 1e-6,
         max_seq: Optional[int] = None, positions: Optional[Sequence[int]] = None,
         k_outlier_frac: float = 0.0, k_outlier_scale: float = 20.0,
         extra_blocks: int = 0, device="cpu", name: str = "custom") -> Workload:
    """Build one decode step's inputs.  lens[b] = L_b (tokens including the new one);
    positions default to L_b - 1.  Paged pools hold exactly sum_b ceil(L_b/64) blocks
    (+ extra_blocks) and the page table maps (b, logical block) in order onto a random
    permutation of the pool."""
    d = HEAD_DIM
    lens = [int(x) for x in lens]
    assert len(lens) == B
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    if max_seq is None:
        max_seq = max(lens)
    seq_lens = torch.tensor(lens, dtype=torch.int32)
    pos = torch.tensor(positions if positions is not None else [L - 1 for L in lens], dtype=torch.int32)
    q_new = _normal_bf16(gen, (B, Hq, d), device)
    k_new = _normal_bf16(gen, (B, Hkv, d), device)
    v_new = _normal_bf16(gen, (B, Hkv, d), device)
    if qk_norm:
        q_norm_w = _normal_bf16(gen, (d,), device, scale=0.1, mean=1.0)
        k_norm_w = _normal_bf16(gen, (d,), device, scale=0.1, mean=1.0)
    else:
        q_norm_w = k_norm_w = None
    if paged:
        nblk_b = [-(-L // BLOCK) for L in lens]
        num_blocks = sum(nblk_b) + int(extra_blocks)
        shape = (num_blocks, BLOCK, Hkv, d)
    else:
        num_blocks = 0
        shape = (B, max_seq, Hkv, d)
    kf = torch.randn(shape, generator=gen, dtype=torch.float32, device=device)
    vf = torch.randn(shape, generator=gen, dtype=torch.float32, device=device)
    if k_outlier_frac > 0.0:
        u = torch.rand(shape, generator=gen, dtype=torch.float32, device=device)
        kf = torch.where(u < k_outlier_frac, kf * k_outlier_scale, kf)
        del u
    k_cache = kf.to(torch.bfloat16)
    del kf
    v_cache = vf.to(torch.bfloat16)
    del vf
    page_table = None
    if paged:
        perm = torch.randperm(num_blocks, generator=gen, device=device).to(torch.int32).cpu()
        mb = -(-max_seq // BLOCK)
        pt = torch.full((B, mb), -1, dtype=torch.int32)
        k = 0
        for b in range(B):
            n = nblk_b[b]
            pt[b, :n] = perm[k:k + n]
            k += n
        page_table = pt.to(device)
    # theta and eps cross the C ABI as binary32; keep exactly the values the library sees
    return Workload(name=name, B=B, Hq=Hq, Hkv=Hkv, d=d, block_size=BLOCK if paged else 0,
                    max_seq=int(max_seq), num_blocks=num_blocks, rope_theta=float(np.float32(rope_theta)),
                    eps=float(np.float32(eps)), q_new=q_new, k_new=k_new, v_new=v_new, k_cache=k_cache,
                    v_cache=v_cache, page_table=page_table, seq_lens=seq_lens.to(device),
                    positions=pos.to(device), q_norm_w=q_norm_w, k_norm_w=k_norm_w)


def ragged_lengths(B: int, lo: int, hi: int, seed: int) -> list:
    """B integer lengths uniform in [lo, hi] inclusive, drawn first from the seed."""
    gen = torch.Generator()
    gen.manual_seed(int(seed))
    return [int(x) for x in torch.randint(lo, hi + 1, (B,), generator=gen)]


WORKLOADS = ("qwen3-14b-tiny", "qwen3-14b-4k", "qwen3-14b-ragged", "llama3-70b-128k", "qwen3-14b-40layer")
LAYERS_40 = 40


def named(name: str, *, device="cpu", seed: int = 0, layer: int = 0) -> Workload:
    """One of the five named decode geometries (one layer of the 40-layer sweep when
    name == 'qwen3-14b-40layer'; layer l draws from seed * 1000 + l)."""
    if name == "qwen3-14b-tiny":
        return make(1, 40, 8, [256], paged=False, seed=seed, rope_theta=1e6, device=device, name=name)
    if name == "qwen3-14b-4k":
        return make(1, 40, 8, [4096], paged=False, seed=seed, rope_theta=1e6, device=device, name=name)
    if name == "qwen3-14b-ragged":
        lens = ragged_lengths(32, 512, 8192, seed)
        return make(32, 40, 8, lens, paged=True, seed=seed, rope_theta=1e6, device=device, name=name)
    if name == "llama3-70b-128k":
        return make(1, 64, 8, [131072], paged=False, seed=seed, qk_norm=False, rope_theta=5e5,
                    device=device, name=name)
    if name == "qwen3-14b-40layer":
        return make(8, 40, 8, [32768] * 8, paged=True, seed=seed * 1000 + layer, rope_theta=1e6,
                    k_outlier_frac=0.01, k_outlier_scale=20.0, device=device, name=f"{name}/layer{layer}")
    raise KeyError(name)


DECODE_STEPS = 64


def decode_sweep(steps: int = DECODE_STEPS, layers: int = LAYERS_40, L_end: int = 4096, *, device="cpu",
                 seed: int = 0) -> list:
    """Autoregressive decode through a stack of `layers` layers of the 4k geometry (B=1,
    40/8 heads, contiguous, QK-norm, theta 1e6, capacity L_end): step t appends the token
    at position L_end - steps + t with fresh q/k/v and attends to the L_end - steps + t + 1
    tokens up to it.  Returns [steps][layers] workloads; the steps of a layer share its
    caches, norm weights and table (layer l's cache draws from seed * 1000 + l, its step
    t inputs from (seed * 1000 + l) * 4096 + t)."""
    base = [make(1, 40, 8, [L_end], paged=False, seed=seed * 1000 + l, rope_theta=1e6, device=device,
                 name=f"qwen3-14b-4k-decode/layer{l}") for l in range(layers)]
    out = []
    for t in range(steps):
        L = L_end - steps + t + 1
        row = []
        for l, w in enumerate(base):
            gen = torch.Generator(device=device)
            gen.manual_seed((seed * 1000 + l) * 4096 + t)
            row.append(dataclasses.replace(
                w, name=f"{w.name}/step{t}",
                q_new=_normal_bf16(gen, (1, w.Hq, w.d), device), k_new=_normal_bf16(gen, (1, w.Hkv, w.d), device),
                v_new=_normal_bf16(gen, (1, w.Hkv, w.d), device),
                seq_lens=torch.tensor([L], dtype=torch.int32, device=device),
                positions=torch.tensor([L - 1], dtype=torch.int32, device=device)))
        out.append(row)
    return out


def kv_bytes_named(name: str, seed: int = 0) -> int:
    """KV bytes one step of a named workload reads (all 40 layers for the sweep)."""
    per_token = 8 * HEAD_DIM * 2 * 2
    if name == "qwen3-14b-tiny":
        return 256 * per_token
    if name == "qwen3-14b-4k":
        return 4096 * per_token
    if name == "qwen3-14b-ragged":
        return sum(ragged_lengths(32, 512, 8192, seed)) * per_token
    if name == "llama3-70b-128k":
        return 131072 * per_token
    if name == "qwen3-14b-40layer":
        return LAYERS_40 * 8 * 32768 * per_token
    raise KeyError(name)


def sample_pairs(B: int, Hq: int, n: int, seed: int) -> np.ndarray:
    """n distinct (b, h) pairs drawn from the seed (for sampled parity at full size)."""
    rng = np.random.default_rng(seed)
    flat = rng.choice(B * Hq, size=min(n, B * Hq), replace=False)
    return np.stack([flat // Hq, flat % Hq], axis=1).astype(np.int32)


def gather_sequence(w: Workload, b: int):
    """K and V rows of sequence b in token order as contiguous [max_seq', H_kv, d] tensors
    (data movement only), for feeding one sequence to the oracle without copying a whole
    pool to the host."""
    L = int(w.seq_lens[b].item())
    if w.paged:
        nb = -(-L // BLOCK)
        pages = w.page_table[b, :nb].long()
        k = w.k_cache.index_select(0, pages).reshape(nb * BLOCK, w.Hkv, w.d)
        v = w.v_cache.index_select(0, pages).reshape(nb * BLOCK, w.Hkv, w.d)
    else:
        k = w.k_cache[b]
        v = w.v_cache[b]
    return k, v


# ----------------------------------------------------------------------------- chunked prefill

@dataclasses.dataclass
class PrefillWorkload:
    """One chunk of causal prefill: T new tokens per sequence at positions
    q_start[b] .. q_start[b] + T - 1 on a cache holding the tokens before them."""
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    T: int
    block_size: int
    max_seq: int
    num_blocks: int
    rope_theta: float
    eps: float
    q_new: torch.Tensor      # [B, T, Hq, d] bf16
    k_new: torch.Tensor      # [B, T, Hkv, d] bf16
    v_new: torch.Tensor      # [B, T, Hkv, d] bf16
    k_cache: torch.Tensor    # paged [nb, 64, Hkv, d] or contiguous [B, max_seq, Hkv, d] bf16
    v_cache: torch.Tensor
    page_table: Optional[torch.Tensor]  # [B, ceil(max_seq/64)] int32
    q_start: torch.Tensor    # [B] int32
    q_norm_w: Optional[torch.Tensor]
    k_norm_w: Optional[torch.Tensor]

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def paged(self) -> bool:
        return self.block_size > 0

    @property
    def num_rows(self) -> int:
        return self.num_blocks * BLOCK if self.paged else self.B * self.max_seq

    def flops(self) -> int:
        """Algorithmic flops of the attention: 4 d per (query head, visible key) pair --
        2 d for q.k and 2 d for p v -- over every chunk token, which sees q_start + i + 1 keys."""
        starts = [int(x) for x in self.q_start.cpu()]
        keys = sum(self.T * s + self.T * (self.T + 1) // 2 for s in starts)
        return 4 * self.d * self.Hq * keys


def make_prefill(B: int, Hq: int, Hkv: int, T: int, q_start: Sequence[int], *, paged: bool, seed: int = 0,
                 qk_norm: bool = True, rope_theta: float = 1e6, eps: float = 1e-6, max_seq: Optional[int] = None,
                 device="cpu", name: str = "custom-prefill") -> PrefillWorkload:
    """Build one prefill chunk's inputs.  Draw order: q/k/v of the chunk, QK-norm weights,
    K cache, V cache, page-table permutation (the same distributions as a decode step).
    Every cache row is drawn, including the chunk's own rows (which the call overwrites)
    and rows past it (which it must never read).  Paged pools hold ceil(max_seq / 64)
    blocks per sequence, mapped in order onto a random permutation of the pool."""
    d = HEAD_DIM
    starts = [int(x) for x in q_start]
    assert len(starts) == B
    if max_seq is None:
        max_seq = max(starts) + T
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    q_new = _normal_bf16(gen, (B, T, Hq, d), device)
    k_new = _normal_bf16(gen, (B, T, Hkv, d), device)
    v_new = _normal_bf16(gen, (B, T, Hkv, d), device)
    if qk_norm:
        q_norm_w = _normal_bf16(gen, (d,), device, scale=0.1, mean=1.0)
        k_norm_w = _normal_bf16(gen, (d,), device, scale=0.1, mean=1.0)
    else:
        q_norm_w = k_norm_w = None
    mb = -(-max_seq // BLOCK)
    if paged:
        num_blocks = B * mb
        shape = (num_blocks, BLOCK, Hkv, d)
    else:
        num_blocks = 0
        shape = (B, max_seq, Hkv, d)
    k_cache = _normal_bf16(gen, shape, device)
    v_cache = _normal_bf16(gen, shape, device)
    page_table = None
    if paged:
        perm = torch.randperm(num_blocks, generator=gen, device=device).to(torch.int32)
        page_table = perm.reshape(B, mb).contiguous()
    return PrefillWorkload(name=name, B=B, Hq=Hq, Hkv=Hkv, d=d, T=int(T), block_size=BLOCK if paged else 0,
                           max_seq=int(max_seq), num_blocks=num_blocks, rope_theta=float(np.float32(rope_theta)),
                           eps=float(np.float32(eps)), q_new=q_new, k_new=k_new, v_new=v_new, k_cache=k_cache,
                           v_cache=v_cache, page_table=page_table,
                           q_start=torch.tensor(starts, dtype=torch.int32, device=device),
                           q_norm_w=q_norm_w, k_norm_w=k_norm_w)


PREFILL_WORKLOADS = ("qwen3-14b-prefill-4k",)


def named_prefill(name: str, *, device="cpu", seed: int = 0) -> PrefillWorkload:
    """``qwen3-14b-prefill-4k``: the last 1024-token chunk of a 4096-token prompt (B=1,
    40/8 heads, contiguous cache of 4096 tokens, QK-norm, theta 1e6): 1024 new tokens at
    positions 3072..4095 over the 3072 cached ones."""
    if name == "qwen3-14b-prefill-4k":
        return make_prefill(1, 40, 8, 1024, [3072], paged=False, seed=seed, max_seq=4096, device=device, name=name)
    raise KeyError(name)


# ----------------------------------------------------------------------------- 4-bit KV cache

@dataclasses.dataclass
class Q4Workload:
    """One decode step over a 4-bit cache (include/gqa_q4.h): the decode step's inputs with
    the cache as packed Lloyd-Max indices [rows, H_kv, 64] (uint8) and one fp32 scale per
    row, the rotation's signs [128] (int8, +-1) and the codebook [16] (bf16)."""
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    block_size: int
    max_seq: int
    num_blocks: int
    rope_theta: float
    eps: float
    q_new: torch.Tensor
    k_new: torch.Tensor
    v_new: torch.Tensor
    k_idx: torch.Tensor      # uint8 [rows, Hkv, 64]
    v_idx: torch.Tensor
    k_scale: torch.Tensor    # float32 [rows, Hkv]
    v_scale: torch.Tensor
    page_table: Optional[torch.Tensor]
    seq_lens: torch.Tensor
    positions: torch.Tensor
    q_norm_w: Optional[torch.Tensor]
    k_norm_w: Optional[torch.Tensor]
    rot_signs: torch.Tensor  # int8 [128]
    codebook: torch.Tensor   # bf16 [16]

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def paged(self) -> bool:
        return self.block_size > 0

    @property
    def num_rows(self) -> int:
        return self.num_blocks * BLOCK if self.paged else self.B * self.max_seq

    def kv_bytes(self) -> int:
        """Bytes of the cache the step reads: per token and KV head, 2 x (64 index bytes +
        a 4-byte scale)."""
        return int(self.seq_lens.long().sum().item()) * self.Hkv * 2 * (64 + 4)


def make_q4(B: int, Hq: int, Hkv: int, lens: Sequence[int], *, paged: bool, seed: int = 0, qk_norm: bool = True,
            rope_theta: float = 1e6, eps: float = 1e-6, max_seq: Optional[int] = None, device="cpu",
            name: str = "custom-q4", codebook_bits: Optional[np.ndarray] = None) -> Q4Workload:
    """The decode step's draws (lengths, q/k/v of the new token, norm weights, page table),
    with the cache drawn directly in its stored form: uniformly random index bytes and
    scales uniform in [0.5, 1.2] (the scale a row of N(0, 1) entries gets), plus random
    rotation signs.  The codebook is the caller's levels (default: the library's
    Lloyd-Max levels, gqa_q4_codebook)."""
    d = HEAD_DIM
    lens = [int(x) for x in lens]
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    if max_seq is None:
        max_seq = max(lens)
    q_new = _normal_bf16(gen, (B, Hq, d), device)
    k_new = _normal_bf16(gen, (B, Hkv, d), device)
    v_new = _normal_bf16(gen, (B, Hkv, d), device)
    if qk_norm:
        q_norm_w = _normal_bf16(gen, (d,), device, scale=0.1, mean=1.0)
        k_norm_w = _normal_bf16(gen, (d,), device, scale=0.1, mean=1.0)
    else:
        q_norm_w = k_norm_w = None
    if paged:
        nblk_b = [-(-L // BLOCK) for L in lens]
        num_blocks = sum(nblk_b)
        rows = num_blocks * BLOCK
    else:
        num_blocks = 0
        rows = B * max_seq
    k_idx = torch.randint(0, 256, (rows, Hkv, d // 2), generator=gen, device=device, dtype=torch.int32).to(torch.uint8)
    v_idx = torch.randint(0, 256, (rows, Hkv, d // 2), generator=gen, device=device, dtype=torch.int32).to(torch.uint8)
    k_scale = torch.rand((rows, Hkv), generator=gen, device=device) * 0.7 + 0.5
    v_scale = torch.rand((rows, Hkv), generator=gen, device=device) * 0.7 + 0.5
    signs = (torch.randint(0, 2, (d,), generator=gen, device=device, dtype=torch.int32) * 2 - 1).to(torch.int8)
    page_table = None
    if paged:
        perm = torch.randperm(num_blocks, generator=gen, device=device).to(torch.int32).cpu()
        mb = -(-max_seq // BLOCK)
        pt = torch.full((B, mb), -1, dtype=torch.int32)
        k = 0
        for b in range(B):
            n = nblk_b[b]
            pt[b, :n] = perm[k:k + n]
            k += n
        page_table = pt.to(device)
    if codebook_bits is None:
        from .binding import q4_codebook
        codebook_bits = q4_codebook()
    codebook = torch.from_numpy(np.asarray(codebook_bits, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)
    return Q4Workload(name=name, B=B, Hq=Hq, Hkv=Hkv, d=d, block_size=BLOCK if paged else 0, max_seq=int(max_seq),
                      num_blocks=num_blocks, rope_theta=float(np.float32(rope_theta)), eps=float(np.float32(eps)),
                      q_new=q_new, k_new=k_new, v_new=v_new, k_idx=k_idx, v_idx=v_idx, k_scale=k_scale,
                      v_scale=v_scale, page_table=page_table,
                      seq_lens=torch.tensor(lens, dtype=torch.int32, device=device),
                      positions=torch.tensor([L - 1 for L in lens], dtype=torch.int32, device=device),
                      q_norm_w=q_norm_w, k_norm_w=k_norm_w, rot_signs=signs, codebook=codebook.to(device))


Q4_WORKLOADS = ("qwen3-14b-4k-q4", "qwen3-14b-ragged-q4")


def named_q4(name: str, *, device="cpu", seed: int = 0) -> Q4Workload:
    """The 4k and ragged decode geometries with a 4-bit cache."""
    if name == "qwen3-14b-4k-q4":
        return make_q4(1, 40, 8, [4096], paged=False, seed=seed, device=device, name=name)
    if name == "qwen3-14b-ragged-q4":
        return make_q4(32, 40, 8, ragged_lengths(32, 512, 8192, seed), paged=True, seed=seed, device=device, name=name)
    raise KeyError(name)
