"""Thin ctypes binding over libgqa_decode.so (include/gqa_decode.h, gqa_prefill.h, gqa_q4.h).

Argument marshalling only: every step of the decode path runs in the library's CUDA
kernels.  Device tensors are torch tensors (device memory and streams come from torch);
host buffers are numpy arrays or CPU torch tensors.  ``load()`` raises if the library
cannot be loaded -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading
from typing import Optional

import numpy as np

from . import build as _build

(GQA_OK, GQA_ERR_INVALID_ARG, GQA_ERR_UNSUPPORTED, GQA_ERR_CUDA, GQA_ERR_WORKSPACE,
 GQA_ERR_SCRATCH_LIMIT) = range(6)
STATIC_SCRATCH_BYTES = 32 << 20
DEVERR_POSITION, DEVERR_SEQLEN, DEVERR_PAGE, DEVERR_TIMEOUT, DEVERR_LAUNCH = 0x1, 0x2, 0x4, 0x8, 0x10
HEADER = os.path.join(_build.ROOT, "include", "gqa_decode.h")
HEADERS = _build.HEADERS

_lock = threading.Lock()
_lib = None


class GqaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


class PlanDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "batch", "num_q_heads", "num_kv_heads", "head_dim", "block_size", "max_seq_len",
        "num_cache_blocks", "num_workers", "device", "cluster_size", "ordered_start")]


class PrefillDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "batch", "num_q_heads", "num_kv_heads", "head_dim", "chunk_len", "block_size", "max_seq_len",
        "num_cache_blocks", "device")]


def header_functions() -> list:
    """Names of the functions the headers under include/ declare."""
    names = set()
    for path in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(path).read(), flags=re.S)
        names.update(re.findall(r"\b(gqa_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def load(build: bool = True):
    """Load the library (building it first when stale); raises on failure."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.build() if build else _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"libgqa_decode.so is missing ({path}); build it with "
                               "gqa_decode_attention_fa_gb300.build.build()")
        lib = ctypes.CDLL(path)
        P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        lib.gqa_plan_create.argtypes = [ctypes.POINTER(PlanDesc), P, ctypes.POINTER(P)]
        lib.gqa_plan_destroy.argtypes = [P]
        lib.gqa_plan_num_workers.argtypes = [P]
        lib.gqa_plan_num_workers.restype = I
        lib.gqa_plan_describe.argtypes = [ctypes.POINTER(PlanDesc), P, I, P, P, P, P]
        lib.gqa_plan_describe.restype = I
        lib.gqa_plan_set_ordered_start.argtypes = [P, I]
        lib.gqa_plan_set_ordered_start.restype = I
        lib.gqa_plan_num_splits.argtypes = [P]
        lib.gqa_plan_num_splits.restype = I
        lib.gqa_plan_cluster_size.argtypes = [P]
        lib.gqa_plan_cluster_size.restype = I
        lib.gqa_plan_workspace_bytes.argtypes = [P]
        lib.gqa_plan_workspace_bytes.restype = ctypes.c_size_t
        step = [P, P, P, P, P, P, P, P, P, P, P, F, F]
        lib.gqa_decode_attn.argtypes = step + [P, P]
        lib.gqa_decode_attn_host.argtypes = step + [P, P]
        lib.gqa_attention_splitkv.argtypes = [P, P, P, P, P, P, P, P, P, P, P, F, F, P]
        lib.gqa_combine.argtypes = [P, P, P, P]
        lib.gqa_plan_read_q_rot.argtypes = [P, P]
        lib.gqa_plan_device_errors.argtypes = [P, ctypes.POINTER(ctypes.c_uint32), I]
        lib.gqa_partition_describe.argtypes = [P, I, I, I, I, P]
        lib.gqa_partition_describe.restype = ctypes.c_longlong
        lib.gqa_decode_attn_static.argtypes = [ctypes.POINTER(PlanDesc)] + step[1:] + [P, P, P]
        lib.gqa_prefill_attn.argtypes = [ctypes.POINTER(PrefillDesc)] + [P] * 9 + [F, F, P, P, P]
        lib.gqa_q4_codebook.argtypes = [P]
        lib.gqa_decode_attn_q4.argtypes = [P] * 15 + [F, F, P, P]
        lib.gqa_status_string.argtypes = [I]
        lib.gqa_status_string.restype = ctypes.c_char_p
        for name in ("gqa_plan_create", "gqa_plan_destroy", "gqa_decode_attn", "gqa_decode_attn_host",
                     "gqa_attention_splitkv", "gqa_combine", "gqa_plan_read_q_rot",
                     "gqa_plan_device_errors", "gqa_decode_attn_static", "gqa_prefill_attn", "gqa_q4_codebook",
                     "gqa_decode_attn_q4"):
            getattr(lib, name).restype = I
        _lib = lib
    return _lib


def status_string(status: int) -> str:
    try:
        return load(build=False).gqa_status_string(int(status)).decode()
    except Exception:  # noqa: BLE001 - only used to format an error message
        return "status"


def _check(status: int, what: str):
    if status != GQA_OK:
        raise GqaError(status, what)


def _dptr(t) -> Optional[int]:
    """Device pointer of a torch tensor (None passes NULL)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _hptr(a) -> Optional[int]:
    """Host pointer of a numpy array or CPU torch tensor."""
    if a is None:
        return None
    if isinstance(a, np.ndarray):
        if not a.flags["C_CONTIGUOUS"]:
            raise ValueError("expected a C-contiguous array")
        return a.ctypes.data
    if a.is_cuda or not a.is_contiguous():
        raise ValueError("expected a contiguous host tensor")
    return a.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return int(stream) if isinstance(stream, int) else stream.cuda_stream


def partition_describe(seq_lens, num_kv_heads: int, max_seq_len: int, num_workers: int):
    """Host view of the split-KV partition: (total tiles, [W, 2] worker ranges)."""
    sl = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
    rng = np.zeros((num_workers, 2), dtype=np.int64)
    T = load().gqa_partition_describe(sl.ctypes.data, len(sl), int(num_kv_heads), int(max_seq_len),
                                      int(num_workers), rng.ctypes.data)
    if T < 0:
        raise ValueError("bad partition arguments")
    return int(T), rng


GB300_SMS = 152
# clusters of 1, 2, ..., 16 single-launch CTAs resident at once on GB300 (cudaOccupancyMaxActiveClusters)
GB300_CLUSTER_CAPACITY = (152, 76, 46, 36, 28, 23, 15, 15, 15, 13, 8, 8, 7, 7, 7, 7)


def plan_describe(batch: int, num_q_heads: int, num_kv_heads: int, max_seq_len: int, *, block_size: int = 0,
                  num_cache_blocks: int = 0, num_workers: int = 0, cluster_size: int = 0, seq_lens_host=None,
                  num_sms: int = GB300_SMS, cluster_capacity=GB300_CLUSTER_CAPACITY, head_dim: int = 128,
                  ordered_start: bool = False):
    """The planner's choices without a GPU (gqa_plan_describe): (workers, cluster size, splits)."""
    desc = PlanDesc(int(batch), int(num_q_heads), int(num_kv_heads), int(head_dim), int(block_size),
                    int(max_seq_len), int(num_cache_blocks), int(num_workers), 0, int(cluster_size),
                    int(bool(ordered_start)))
    sl = None if seq_lens_host is None else np.ascontiguousarray(np.asarray(seq_lens_host, dtype=np.int32))
    cap = np.ascontiguousarray(np.asarray(cluster_capacity, dtype=np.int32))
    if cap.shape != (16,):
        raise ValueError("cluster_capacity: 16 counts, for clusters of 1 .. 16 CTAs")
    out = np.zeros(3, dtype=np.int32)
    _check(load().gqa_plan_describe(ctypes.byref(desc), None if sl is None else sl.ctypes.data, int(num_sms),
                                    cap.ctypes.data, out[0:].ctypes.data, out[1:].ctypes.data,
                                    out[2:].ctypes.data), "gqa_plan_describe")
    return int(out[0]), int(out[1]), int(out[2])


def decode_attn_static(batch: int, num_q_heads: int, num_kv_heads: int, max_seq_len: int, q_new, k_new, v_new,
                       k_cache, v_cache, page_table, seq_lens, positions, q_norm_w, k_norm_w, rope_theta: float,
                       eps: float, out, *, block_size: int = 0, num_cache_blocks: int = 0, head_dim: int = 128,
                       num_workers: int = 0, cluster_size: int = 0, device: int = 0, device_errors=None,
                       stream=None, ordered_start: bool = False):
    """One decode step through gqa_decode_attn_static: no plan, no device allocation; the
    workspace is the library's fixed static scratch of the device.  `device_errors` is an
    optional int32/uint32 device tensor of one element the kernels OR error bits into."""
    desc = PlanDesc(int(batch), int(num_q_heads), int(num_kv_heads), int(head_dim), int(block_size),
                    int(max_seq_len), int(num_cache_blocks), int(num_workers), int(device), int(cluster_size),
                    int(bool(ordered_start)))
    _check(load().gqa_decode_attn_static(
        ctypes.byref(desc), _dptr(q_new), _dptr(k_new), _dptr(v_new), _dptr(k_cache), _dptr(v_cache),
        _dptr(page_table), _dptr(seq_lens), _dptr(positions), _dptr(q_norm_w), _dptr(k_norm_w), float(rope_theta),
        float(eps), _dptr(out), _dptr(device_errors), _stream(stream)), "gqa_decode_attn_static")


def decode_attn_static_workload(w, out, *, num_workers: int = 0, cluster_size: int = 0, device: int = 0,
                                device_errors=None, stream=None):
    """gqa_decode_attn_static on a workload's tensors (see workloads.Workload)."""
    decode_attn_static(w.B, w.Hq, w.Hkv, w.max_seq, w.q_new, w.k_new, w.v_new, w.k_cache, w.v_cache, w.page_table,
                       w.seq_lens, w.positions, w.q_norm_w, w.k_norm_w, w.rope_theta, w.eps, out,
                       block_size=w.block_size, num_cache_blocks=w.num_blocks, num_workers=num_workers,
                       cluster_size=cluster_size, device=device, device_errors=device_errors, stream=stream)


def prefill_attn(batch: int, num_q_heads: int, num_kv_heads: int, chunk_len: int, max_seq_len: int, q_new, k_new,
                 v_new, k_cache, v_cache, page_table, q_start, q_norm_w, k_norm_w, rope_theta: float, eps: float, out,
                 *, block_size: int = 0, num_cache_blocks: int = 0, head_dim: int = 128, device: int = 0,
                 device_errors=None, stream=None):
    """One chunk of causal prefill through gqa_prefill_attn (include/gqa_prefill.h)."""
    desc = PrefillDesc(int(batch), int(num_q_heads), int(num_kv_heads), int(head_dim), int(chunk_len),
                       int(block_size), int(max_seq_len), int(num_cache_blocks), int(device))
    _check(load().gqa_prefill_attn(
        ctypes.byref(desc), _dptr(q_new), _dptr(k_new), _dptr(v_new), _dptr(k_cache), _dptr(v_cache),
        _dptr(page_table), _dptr(q_start), _dptr(q_norm_w), _dptr(k_norm_w), float(rope_theta), float(eps),
        _dptr(out), _dptr(device_errors), _stream(stream)), "gqa_prefill_attn")


def prefill_attn_workload(w, out, *, device: int = 0, device_errors=None, stream=None):
    """gqa_prefill_attn on a prefill workload's tensors (see workloads.PrefillWorkload)."""
    prefill_attn(w.B, w.Hq, w.Hkv, w.T, w.max_seq, w.q_new, w.k_new, w.v_new, w.k_cache, w.v_cache, w.page_table,
                 w.q_start, w.q_norm_w, w.k_norm_w, w.rope_theta, w.eps, out, block_size=w.block_size,
                 num_cache_blocks=w.num_blocks, device=device, device_errors=device_errors, stream=stream)


def q4_codebook() -> np.ndarray:
    """The 16 Lloyd-Max levels of N(0,1) as bf16 bit patterns (gqa_q4_codebook)."""
    out = np.zeros(16, dtype=np.uint16)
    _check(load().gqa_q4_codebook(out.ctypes.data), "gqa_q4_codebook")
    return out


class Plan:
    """A gqa_plan_t: geometry, split-worker count and the workspace (allocated once)."""

    def __init__(self, batch: int, num_q_heads: int, num_kv_heads: int, max_seq_len: int, *,
                 block_size: int = 0, num_cache_blocks: int = 0, head_dim: int = 128, num_workers: int = 0,
                 device: int = 0, seq_lens_host=None, cluster_size: int = 0, ordered_start: bool = False):
        self._lib = load()
        self.desc = PlanDesc(int(batch), int(num_q_heads), int(num_kv_heads), int(head_dim), int(block_size),
                             int(max_seq_len), int(num_cache_blocks), int(num_workers), int(device),
                             int(cluster_size), int(bool(ordered_start)))
        sl = None
        if seq_lens_host is not None:
            sl = np.ascontiguousarray(np.asarray(seq_lens_host, dtype=np.int32))
        self._h = ctypes.c_void_p()
        _check(self._lib.gqa_plan_create(ctypes.byref(self.desc), None if sl is None else sl.ctypes.data,
                                         ctypes.byref(self._h)), "gqa_plan_create")

    @classmethod
    def for_workload(cls, w, num_workers: int = 0, device: int = 0, cluster_size: int = 0) -> "Plan":
        return cls(w.B, w.Hq, w.Hkv, w.max_seq, block_size=w.block_size, num_cache_blocks=w.num_blocks,
                   num_workers=num_workers, device=device, seq_lens_host=w.seq_lens.cpu().numpy(),
                   cluster_size=cluster_size)

    def close(self):
        if getattr(self, "_h", None) and self._h.value:
            _check(self._lib.gqa_plan_destroy(self._h), "gqa_plan_destroy")
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:  # noqa: BLE001 - interpreter shutdown
            pass

    @property
    def handle(self):
        return self._h

    @property
    def num_workers(self) -> int:
        return self._lib.gqa_plan_num_workers(self._h)

    def set_ordered_start(self, ordered: bool = True):
        """Launch each step's first kernel in plain stream order (gqa_plan_set_ordered_start)."""
        _check(self._lib.gqa_plan_set_ordered_start(self._h, int(bool(ordered))), "gqa_plan_set_ordered_start")

    @property
    def num_splits(self) -> int:
        return self._lib.gqa_plan_num_splits(self._h)

    @property
    def cluster_size(self) -> int:
        """The single-launch form's cluster size, 0 for split-KV + combine."""
        return self._lib.gqa_plan_cluster_size(self._h)

    @property
    def workspace_bytes(self) -> int:
        return self._lib.gqa_plan_workspace_bytes(self._h)

    # ------------------------------------------------------------------ the step
    def decode_attn(self, q_new, k_new, v_new, k_cache, v_cache, page_table, seq_lens, positions,
                    q_norm_w, k_norm_w, rope_theta: float, eps: float, out, stream=None):
        _check(self._lib.gqa_decode_attn(
            self._h, _dptr(q_new), _dptr(k_new), _dptr(v_new), _dptr(k_cache), _dptr(v_cache), _dptr(page_table),
            _dptr(seq_lens), _dptr(positions), _dptr(q_norm_w), _dptr(k_norm_w), float(rope_theta), float(eps),
            _dptr(out), _stream(stream)), "gqa_decode_attn")

    def decode_attn_host(self, q_new, k_new, v_new, k_cache, v_cache, page_table, seq_lens, positions,
                         q_norm_w, k_norm_w, rope_theta: float, eps: float, out, stream=None):
        """q/k/v_new, seq_lens, positions and out are host buffers; caches, page table and
        norm weights are device tensors.  Synchronise the stream before reading `out`."""
        _check(self._lib.gqa_decode_attn_host(
            self._h, _hptr(q_new), _hptr(k_new), _hptr(v_new), _dptr(k_cache), _dptr(v_cache), _dptr(page_table),
            _hptr(seq_lens), _hptr(positions), _dptr(q_norm_w), _dptr(k_norm_w), float(rope_theta), float(eps),
            _hptr(out), _stream(stream)), "gqa_decode_attn_host")

    def attention_splitkv(self, q_new, k_new, v_new, k_cache, v_cache, page_table, seq_lens, positions, q_norm_w,
                          k_norm_w, rope_theta: float, eps: float, stream=None):
        _check(self._lib.gqa_attention_splitkv(
            self._h, _dptr(q_new), _dptr(k_new), _dptr(v_new), _dptr(k_cache), _dptr(v_cache), _dptr(page_table),
            _dptr(seq_lens), _dptr(positions), _dptr(q_norm_w), _dptr(k_norm_w), float(rope_theta), float(eps),
            _stream(stream)), "gqa_attention_splitkv")

    def combine(self, seq_lens, out, stream=None):
        _check(self._lib.gqa_combine(self._h, _dptr(seq_lens), _dptr(out), _stream(stream)), "gqa_combine")

    def read_q_rot(self) -> np.ndarray:
        d = self.desc
        out = np.zeros((d.batch, d.num_q_heads, d.head_dim), dtype=np.uint16)
        _check(self._lib.gqa_plan_read_q_rot(self._h, out.ctypes.data), "gqa_plan_read_q_rot")
        return out

    def device_errors(self, clear: bool = True) -> int:
        f = ctypes.c_uint32(0)
        _check(self._lib.gqa_plan_device_errors(self._h, ctypes.byref(f), int(bool(clear))), "gqa_plan_device_errors")
        return int(f.value)

    # ------------------------------------------------------------------ convenience
    def decode_attn_q4(self, q_new, k_new, v_new, k_idx, v_idx, k_scale, v_scale, page_table, seq_lens,
                       positions, q_norm_w, k_norm_w, rot_signs, codebook, rope_theta: float, eps: float, out,
                       stream=None):
        """The decode step over a 4-bit cache (gqa_decode_attn_q4, include/gqa_q4.h)."""
        _check(load().gqa_decode_attn_q4(
            self._h, _dptr(q_new), _dptr(k_new), _dptr(v_new), _dptr(k_idx), _dptr(v_idx), _dptr(k_scale),
            _dptr(v_scale), _dptr(page_table), _dptr(seq_lens), _dptr(positions), _dptr(q_norm_w), _dptr(k_norm_w),
            _dptr(rot_signs), _dptr(codebook), float(rope_theta), float(eps), _dptr(out), _stream(stream)),
            "gqa_decode_attn_q4")

    def run_q4(self, w, out, stream=None):
        """gqa_decode_attn_q4 on a 4-bit-cache workload (workloads.Q4Workload)."""
        self.decode_attn_q4(w.q_new, w.k_new, w.v_new, w.k_idx, w.v_idx, w.k_scale, w.v_scale, w.page_table,
                            w.seq_lens, w.positions, w.q_norm_w, w.k_norm_w, w.rot_signs, w.codebook, w.rope_theta,
                            w.eps, out, stream)

    def run(self, w, out, stream=None):
        """One decode step of a workloads.Workload already on this device."""
        self.decode_attn(w.q_new, w.k_new, w.v_new, w.k_cache, w.v_cache, w.page_table, w.seq_lens, w.positions,
                         w.q_norm_w, w.k_norm_w, w.rope_theta, w.eps, out, stream)

    def run_steps(self, w, out, stream=None, between=None):
        """The same step as its two launches; between(i) is called before (i = 0) and
        after (i = 1) the attention launch -- e.g. to record CUDA events around it."""
        if between:
            between(0)
        self.attention_splitkv(w.q_new, w.k_new, w.v_new, w.k_cache, w.v_cache, w.page_table, w.seq_lens,
                               w.positions, w.q_norm_w, w.k_norm_w, w.rope_theta, w.eps, stream)
        if between:
            between(1)
        self.combine(w.seq_lens, out, stream)
