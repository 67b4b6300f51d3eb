"""fp64 CPU oracle for the fused GQA decode-attention step -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this package.  The library (``gqa_decode_attention_fa_gb300``) never does, and the two
share no code: the oracle is plain C (``gqa_oracle.c``) compiled with gcc, wrapped here with
ctypes and numpy for argument marshalling only.

Every tensor crosses this boundary as raw bf16 bit patterns (``numpy.uint16``) or int32
indices, exactly the bits the CUDA path receives.  Results are fp64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gqa_oracle.c")
_LIB = os.path.join(_HERE, "libgqa_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle into ``libgqa_oracle.so`` (gcc, OpenMP, no FP contraction so the
    result is the same on x86-64 and aarch64)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call([
            "gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
            "-fPIC", "-shared", "-o", tmp, _SRC, "-lm",
        ])
        os.replace(tmp, _LIB)
    return _LIB


class Geom(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int), ("d", ctypes.c_int),
        ("block_size", ctypes.c_int), ("max_seq", ctypes.c_int), ("num_rows", ctypes.c_longlong),
    ]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_double.restype = ctypes.c_double
            lib.oracle_round_bf16.argtypes = [ctypes.c_double]
            lib.oracle_round_bf16.restype = ctypes.c_uint16
            lib.oracle_rmsnorm.argtypes = [P, P, ctypes.c_int, ctypes.c_double, P]
            lib.oracle_rope.argtypes = [P, ctypes.c_int, ctypes.c_longlong, ctypes.c_double, P]
            lib.oracle_prologue.argtypes = [ctypes.POINTER(Geom)] + [P] * 10 + [ctypes.c_double, ctypes.c_double, P]
            lib.oracle_prologue.restype = ctypes.c_int
            lib.oracle_attention.argtypes = [ctypes.POINTER(Geom), P, P, P, P, P, P, ctypes.c_int, P]
            lib.oracle_attention.restype = ctypes.c_int
            lib.oracle_attention_streaming.argtypes = [
                ctypes.POINTER(Geom), P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                P, ctypes.c_int, P]
            lib.oracle_prefill_prologue.argtypes = [ctypes.POINTER(Geom), ctypes.c_int] + [P] * 9 + [
                ctypes.c_double, ctypes.c_double, P]
            lib.oracle_prefill_prologue.restype = ctypes.c_int
            lib.oracle_prefill_attention.argtypes = [ctypes.POINTER(Geom), ctypes.c_int, P, P, P, P, P, P,
                                                     ctypes.c_int, P]
            lib.oracle_prefill_attention.restype = ctypes.c_int
            lib.oracle_prefill_blocked.argtypes = [ctypes.POINTER(Geom), ctypes.c_int, P, P, P, P, P,
                                                   ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, P]
            lib.oracle_lloyd_max.argtypes = [ctypes.c_int, P, P]
            lib.oracle_lloyd_max.restype = ctypes.c_int
            lib.oracle_rotate.argtypes = [P, P, ctypes.c_int, P]
            lib.oracle_unrotate.argtypes = [P, P, ctypes.c_int, P]
            lib.oracle_q4_quantize.argtypes = [P, P, P, ctypes.c_int, P, P]
            lib.oracle_q4_dequantize.argtypes = [P, ctypes.c_double, P, P, ctypes.c_int, P]
            lib.oracle_q4_decode_step.argtypes = [ctypes.POINTER(Geom)] + [P] * 12 + [
                ctypes.c_double, ctypes.c_double, P, P, P, ctypes.c_int, P, P]
            lib.oracle_q4_decode_step.restype = ctypes.c_int
            lib.oracle_q4_attention.argtypes = [ctypes.POINTER(Geom)] + [P] * 10 + [P, ctypes.c_int, P]
            lib.oracle_set_threads.argtypes = [ctypes.c_int]
            lib.oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def geom(B, Hq, Hkv, d, block_size, max_seq, num_rows) -> Geom:
    return Geom(int(B), int(Hq), int(Hkv), int(d), int(block_size), int(max_seq), int(num_rows))


# ----------------------------------------------------------------------------- scalars

def bf16_to_f64(bits) -> np.ndarray:
    bits = np.asarray(bits, dtype=np.uint16)
    lib = _load()
    flat = bits.reshape(-1)
    return np.array([lib.oracle_bf16_to_double(int(b)) for b in flat], dtype=np.float64).reshape(bits.shape)


def round_bf16(x) -> np.ndarray:
    """Round fp64 values to bf16 bit patterns (nearest, ties to even), one at a time."""
    x = np.asarray(x, dtype=np.float64)
    lib = _load()
    flat = x.reshape(-1)
    return np.array([lib.oracle_round_bf16(float(v)) for v in flat], dtype=np.uint16).reshape(x.shape)


def rmsnorm(x, w, eps: float) -> np.ndarray:
    x = _c(x, np.float64)
    w = _c(w, np.float64)
    y = np.empty_like(x)
    _load().oracle_rmsnorm(_ptr(x), _ptr(w), x.shape[0], float(eps), _ptr(y))
    return y


def rope(y, pos: int, theta: float) -> np.ndarray:
    y = _c(y, np.float64)
    z = np.empty_like(y)
    _load().oracle_rope(_ptr(y), y.shape[0], int(pos), float(theta), _ptr(z))
    return z


# ----------------------------------------------------------------------------- step

def prologue(g: Geom, q_new, k_new, v_new, k_cache, v_cache, page_table, seq_lens, positions,
             q_norm_w, k_norm_w, rope_theta: float, eps: float):
    """Returns (q_rot bits [B,Hq,d], k_cache', v_cache', status).  The input caches are not
    modified; the returned ones are copies with the new rows written."""
    q_new, k_new, v_new = (_c(a, np.uint16) for a in (q_new, k_new, v_new))
    kc = np.array(k_cache, dtype=np.uint16, copy=True, order="C")
    vc = np.array(v_cache, dtype=np.uint16, copy=True, order="C")
    pt = _c(page_table, np.int32)
    sl, pos = _c(seq_lens, np.int32), _c(positions, np.int32)
    qw, kw = _c(q_norm_w, np.uint16), _c(k_norm_w, np.uint16)
    q_rot = np.zeros((g.B, g.Hq, g.d), dtype=np.uint16)
    st = _load().oracle_prologue(ctypes.byref(g), _ptr(q_new), _ptr(k_new), _ptr(v_new), _ptr(kc), _ptr(vc),
                                 _ptr(pt), _ptr(sl), _ptr(pos), _ptr(qw), _ptr(kw),
                                 float(rope_theta), float(eps), _ptr(q_rot))
    return q_rot, kc, vc, st


def attention(g: Geom, q_rot, k_cache, v_cache, page_table, seq_lens, pairs=None, threads: int | None = None):
    """Brute-force attention in fp64.  Returns (out, threads_used); out is [B,Hq,d], or
    [len(pairs), d] when a list of (b, h) pairs is given."""
    lib = _load()
    if threads:
        lib.oracle_set_threads(int(threads))
    q_rot, kc, vc = (_c(a, np.uint16) for a in (q_rot, k_cache, v_cache))
    pt, sl = _c(page_table, np.int32), _c(seq_lens, np.int32)
    if pairs is not None:
        pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
        out = np.zeros((pr.shape[0], g.d), dtype=np.float64)
        used = lib.oracle_attention(ctypes.byref(g), _ptr(q_rot), _ptr(kc), _ptr(vc), _ptr(pt), _ptr(sl),
                                    _ptr(pr), pr.shape[0], _ptr(out))
    else:
        out = np.zeros((g.B, g.Hq, g.d), dtype=np.float64)
        used = lib.oracle_attention(ctypes.byref(g), _ptr(q_rot), _ptr(kc), _ptr(vc), _ptr(pt), _ptr(sl),
                                    None, 0, _ptr(out))
    return out, used


def attention_streaming(g: Geom, q_rot, k_cache, v_cache, page_table, L: int, b: int, h: int,
                        tile: int, split_bounds) -> np.ndarray:
    q_rot, kc, vc = (_c(a, np.uint16) for a in (q_rot, k_cache, v_cache))
    pt = _c(page_table, np.int32)
    sb = np.ascontiguousarray(np.asarray(split_bounds, dtype=np.int32))
    out = np.zeros(g.d, dtype=np.float64)
    _load().oracle_attention_streaming(ctypes.byref(g), _ptr(q_rot), _ptr(kc), _ptr(vc), _ptr(pt),
                                       int(L), int(b), int(h), int(tile), _ptr(sb), len(sb) - 1, _ptr(out))
    return out


def decode_step(g: Geom, q_new, k_new, v_new, k_cache, v_cache, page_table, seq_lens, positions,
                q_norm_w, k_norm_w, rope_theta: float, eps: float, pairs=None, threads: int | None = None):
    """The whole step: prologue (cache append) then attention over the updated cache.
    Returns dict(out, q_rot, k_cache, v_cache, status, threads)."""
    q_rot, kc, vc, st = prologue(g, q_new, k_new, v_new, k_cache, v_cache, page_table, seq_lens,
                                 positions, q_norm_w, k_norm_w, rope_theta, eps)
    out, used = attention(g, q_rot, kc, vc, page_table, seq_lens, pairs=pairs, threads=threads)
    return dict(out=out, q_rot=q_rot, k_cache=kc, v_cache=vc, status=st, threads=used)


# ----------------------------------------------------------------------------- chunked prefill

def prefill_prologue(g: Geom, T: int, q_new, k_new, v_new, k_cache, v_cache, page_table, q_start,
                     q_norm_w, k_norm_w, rope_theta: float, eps: float):
    """The per-token prologue of a chunk of T tokens per sequence.  q_new [B,T,Hq,d],
    k_new/v_new [B,T,Hkv,d] bits; q_start [B].  Returns (q_rot bits [B,T,Hq,d], k_cache',
    v_cache', status); the input caches are not modified."""
    q_new, k_new, v_new = (_c(a, np.uint16) for a in (q_new, k_new, v_new))
    kc = np.array(k_cache, dtype=np.uint16, copy=True, order="C")
    vc = np.array(v_cache, dtype=np.uint16, copy=True, order="C")
    pt, qs = _c(page_table, np.int32), _c(q_start, np.int32)
    qw, kw = _c(q_norm_w, np.uint16), _c(k_norm_w, np.uint16)
    q_rot = np.zeros((g.B, int(T), g.Hq, g.d), dtype=np.uint16)
    st = _load().oracle_prefill_prologue(ctypes.byref(g), int(T), _ptr(q_new), _ptr(k_new), _ptr(v_new),
                                         _ptr(kc), _ptr(vc), _ptr(pt), _ptr(qs), _ptr(qw), _ptr(kw),
                                         float(rope_theta), float(eps), _ptr(q_rot))
    return q_rot, kc, vc, st


def prefill_attention(g: Geom, T: int, q_rot, k_cache, v_cache, page_table, q_start, triples=None,
                      threads: int | None = None):
    """Causal attention of the chunk, brute force, fp64.  Returns (out, threads_used); out is
    [B,T,Hq,d], or [len(triples), d] for a list of (b, i, h) triples."""
    lib = _load()
    if threads:
        lib.oracle_set_threads(int(threads))
    q_rot, kc, vc = (_c(a, np.uint16) for a in (q_rot, k_cache, v_cache))
    pt, qs = _c(page_table, np.int32), _c(q_start, np.int32)
    if triples is not None:
        tr = np.ascontiguousarray(np.asarray(triples, dtype=np.int32).reshape(-1, 3))
        out = np.zeros((tr.shape[0], g.d), dtype=np.float64)
        used = lib.oracle_prefill_attention(ctypes.byref(g), int(T), _ptr(q_rot), _ptr(kc), _ptr(vc), _ptr(pt),
                                            _ptr(qs), _ptr(tr), tr.shape[0], _ptr(out))
    else:
        out = np.zeros((g.B, int(T), g.Hq, g.d), dtype=np.float64)
        used = lib.oracle_prefill_attention(ctypes.byref(g), int(T), _ptr(q_rot), _ptr(kc), _ptr(vc), _ptr(pt),
                                            _ptr(qs), None, 0, _ptr(out))
    return out, used


def prefill_blocked(g: Geom, T: int, q_rot, k_cache, v_cache, page_table, q_start, b: int, h: int,
                    q_block: int, kv_tile: int) -> np.ndarray:
    """The past / partial / future tile-class form for one (b, h); returns [T, d]."""
    q_rot, kc, vc = (_c(a, np.uint16) for a in (q_rot, k_cache, v_cache))
    pt, qs = _c(page_table, np.int32), _c(q_start, np.int32)
    out = np.zeros((int(T), g.d), dtype=np.float64)
    _load().oracle_prefill_blocked(ctypes.byref(g), int(T), _ptr(q_rot), _ptr(kc), _ptr(vc), _ptr(pt), _ptr(qs),
                                   int(b), int(h), int(q_block), int(kv_tile), _ptr(out))
    return out


def prefill_step(g: Geom, T: int, q_new, k_new, v_new, k_cache, v_cache, page_table, q_start,
                 q_norm_w, k_norm_w, rope_theta: float, eps: float, triples=None, threads: int | None = None):
    """The whole chunk: prologue (T cache rows per sequence) then causal attention.
    Returns dict(out, q_rot, k_cache, v_cache, status, threads)."""
    q_rot, kc, vc, st = prefill_prologue(g, T, q_new, k_new, v_new, k_cache, v_cache, page_table, q_start,
                                         q_norm_w, k_norm_w, rope_theta, eps)
    out, used = prefill_attention(g, T, q_rot, kc, vc, page_table, q_start, triples=triples, threads=threads)
    return dict(out=out, q_rot=q_rot, k_cache=kc, v_cache=vc, status=st, threads=used)


# ----------------------------------------------------------------------------- 4-bit KV cache

def lloyd_max(levels: int = 16):
    """(levels ascending, thresholds, iterations) of the Lloyd-Max quantizer of N(0,1)."""
    lv = np.zeros(levels)
    thr = np.zeros(levels - 1)
    it = _load().oracle_lloyd_max(int(levels), _ptr(lv), _ptr(thr))
    return lv, thr, it


def rotate(x, signs) -> np.ndarray:
    x = _c(x, np.float64)
    sg = _c(signs, np.int8)
    y = np.empty_like(x)
    _load().oracle_rotate(_ptr(x), _ptr(sg), x.shape[0], _ptr(y))
    return y


def unrotate(y, signs) -> np.ndarray:
    y = _c(y, np.float64)
    sg = _c(signs, np.int8)
    x = np.empty_like(y)
    _load().oracle_unrotate(_ptr(y), _ptr(sg), y.shape[0], _ptr(x))
    return x


def q4_quantize(x, signs, codebook_bits):
    """(packed uint8[d/2], sigma) of one row."""
    x = _c(x, np.float64)
    sg, cb = _c(signs, np.int8), _c(codebook_bits, np.uint16)
    packed = np.zeros(x.shape[0] // 2, dtype=np.uint8)
    sigma = ctypes.c_double()
    _load().oracle_q4_quantize(_ptr(x), _ptr(sg), _ptr(cb), x.shape[0], _ptr(packed), ctypes.byref(sigma))
    return packed, sigma.value


def q4_dequantize(packed, sigma: float, signs, codebook_bits) -> np.ndarray:
    pk = _c(packed, np.uint8)
    sg, cb = _c(signs, np.int8), _c(codebook_bits, np.uint16)
    x = np.zeros(pk.shape[0] * 2)
    _load().oracle_q4_dequantize(_ptr(pk), float(sigma), _ptr(sg), _ptr(cb), x.shape[0], _ptr(x))
    return x


def q4_decode_step(g: Geom, q_new, k_new, v_new, k_idx, v_idx, k_scale, v_scale, page_table, seq_lens, positions,
                   q_norm_w, k_norm_w, rope_theta: float, eps: float, signs, codebook_bits, pairs=None):
    """The decode step over a 4-bit cache.  Returns dict(out, q_rot, k_idx, v_idx, k_scale,
    v_scale, status); the input caches are not modified."""
    q_new, k_new, v_new = (_c(a, np.uint16) for a in (q_new, k_new, v_new))
    ki = np.array(k_idx, dtype=np.uint8, copy=True, order="C")
    vi = np.array(v_idx, dtype=np.uint8, copy=True, order="C")
    ks = np.array(k_scale, dtype=np.float32, copy=True, order="C")
    vs = np.array(v_scale, dtype=np.float32, copy=True, order="C")
    pt, sl, pos = _c(page_table, np.int32), _c(seq_lens, np.int32), _c(positions, np.int32)
    qw, kw = _c(q_norm_w, np.uint16), _c(k_norm_w, np.uint16)
    sg, cb = _c(signs, np.int8), _c(codebook_bits, np.uint16)
    q_rot = np.zeros((g.B, g.Hq, g.d), dtype=np.uint16)
    if pairs is not None:
        pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
        out = np.zeros((pr.shape[0], g.d))
        npairs = pr.shape[0]
    else:
        pr, npairs = None, 0
        out = np.zeros((g.B, g.Hq, g.d))
    st = _load().oracle_q4_decode_step(ctypes.byref(g), _ptr(q_new), _ptr(k_new), _ptr(v_new), _ptr(ki), _ptr(vi),
                                       _ptr(ks), _ptr(vs), _ptr(pt), _ptr(sl), _ptr(pos), _ptr(qw), _ptr(kw),
                                       float(rope_theta), float(eps), _ptr(sg), _ptr(cb), _ptr(pr), npairs,
                                       _ptr(q_rot), _ptr(out))
    return dict(out=out, q_rot=q_rot, k_idx=ki, v_idx=vi, k_scale=ks, v_scale=vs, status=st)


def q4_attention(g: Geom, q_rot, k_idx, v_idx, k_scale, v_scale, page_table, seq_lens, signs, codebook_bits,
                 pairs=None) -> np.ndarray:
    """Attention over a given 4-bit cache (no prologue): [B,Hq,d], or [len(pairs), d]."""
    q_rot = _c(q_rot, np.uint16)
    ki, vi = _c(k_idx, np.uint8), _c(v_idx, np.uint8)
    ks, vs = _c(k_scale, np.float32), _c(v_scale, np.float32)
    pt, sl = _c(page_table, np.int32), _c(seq_lens, np.int32)
    sg, cb = _c(signs, np.int8), _c(codebook_bits, np.uint16)
    if pairs is not None:
        pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
        out = np.zeros((pr.shape[0], g.d))
        npairs = pr.shape[0]
    else:
        pr, npairs = None, 0
        out = np.zeros((g.B, g.Hq, g.d))
    _load().oracle_q4_attention(ctypes.byref(g), _ptr(q_rot), _ptr(ki), _ptr(vi), _ptr(ks), _ptr(vs), _ptr(pt),
                                _ptr(sl), None, _ptr(sg), _ptr(cb), _ptr(pr), npairs, _ptr(out))
    return out


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))
