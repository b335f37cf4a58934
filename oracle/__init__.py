"""The oracle: a plain fp64 CPU definition of block-sparse retrieval decode.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` import this package.  The product path (the CUDA
library and its Python binding) never imports it, and the two share no code.

The arithmetic lives in ``srkv_oracle.c`` (plain C, fp64, scalar loops, one
library sort); this module only compiles it with gcc, marshals numpy arrays and
reads results back.  See the header of ``srkv_oracle.c`` for the pages followed
and the readings taken where they are silent.

Inputs follow the layouts of the method on the pages:
  q            [B][Hq][d]            bf16 (as uint16 bit patterns) or float32
  k/v caches   [P][Hkv][S][d]        same dtype as q, or (dtype 2) E4M3 codes (uint8) with
                                     fp32 scales [P][Hkv][S] per row, q then bf16
  block_table  [B][max_blocks] int32 logical block -> physical page
  seq_lens     [B] int32             tokens in the cache (current token included)
  prompt_lens  [B] int32             prefill length, compared with DENSE_BOUNDARY
A configuration is a mapping with the keys of :data:`CFG_KEYS`.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Mapping, Sequence

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "srkv_oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libsrkv_oracle.so")

CFG_KEYS = ("num_q_heads", "num_kv_heads", "head_dim", "block_size", "init_tokens",
            "local_tokens", "topk_percent", "dense_boundary", "dtype")

_ERRORS = {-1: "bad argument", -2: "page id out of range", -3: "out of memory",
           -4: "selection larger than kmax"}


class _Cfg(ctypes.Structure):
    _fields_ = [("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("init_tokens", ctypes.c_int32), ("local_tokens", ctypes.c_int32),
                ("topk_percent", ctypes.c_double), ("dense_boundary", ctypes.c_int32),
                ("dtype", ctypes.c_int32)]


class _Inputs(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k_cache", ctypes.c_void_p),
                ("v_cache", ctypes.c_void_p), ("num_pages", ctypes.c_int64),
                ("block_table", ctypes.c_void_p), ("max_blocks", ctypes.c_int32),
                ("seq_lens", ctypes.c_void_p), ("prompt_lens", ctypes.c_void_p),
                ("batch", ctypes.c_int32), ("k_scale", ctypes.c_void_p),
                ("v_scale", ctypes.c_void_p)]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no FP contraction) into ``oracle/_build``."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(LIB_PATH)
            and os.path.getmtime(LIB_PATH) >= os.path.getmtime(SRC)):
        return LIB_PATH
    tmp = LIB_PATH + f".{os.getpid()}.tmp"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC",
                           "-shared", "-o", tmp, SRC, "-lm", "-lpthread"])
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


_lib = None


def load() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.oracle_kv_cache_bytes.restype = ctypes.c_double
        lib.oracle_kv_cache_bytes.argtypes = [ctypes.c_double] * 5
        lib.oracle_topk_count.restype = ctypes.c_int64
        lib.oracle_topk_count.argtypes = [ctypes.c_int64, ctypes.c_double]
        lib.oracle_num_candidates.restype = ctypes.c_int64
        lib.oracle_num_candidates.argtypes = [ctypes.c_int64, ctypes.c_int32,
                                              ctypes.c_int32, ctypes.c_int32]
        lib.oracle_block_reps.restype = ctypes.c_int
        lib.oracle_e4m3_value.restype = ctypes.c_double
        lib.oracle_e4m3_value.argtypes = [ctypes.c_uint32]
        lib.oracle_e4m3_code.restype = ctypes.c_uint32
        lib.oracle_e4m3_code.argtypes = [ctypes.c_double]
        lib.oracle_quantize_e4m3.restype = ctypes.c_int
        lib.oracle_unit.restype = ctypes.c_int
        lib.oracle_decode_units.restype = ctypes.c_int
        _lib = lib
    return _lib


def _check(rc: int) -> None:
    if rc != 0:
        raise ValueError(f"oracle: {_ERRORS.get(rc, rc)}")


def _cfg(cfg: Mapping) -> _Cfg:
    return _Cfg(*[cfg[k] for k in CFG_KEYS])


def _ptr(a: np.ndarray | None) -> ctypes.c_void_p | None:
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _values(a, dtype: int) -> np.ndarray:
    """bf16 inputs travel as uint16 bit patterns, fp32 as float32, E4M3 codes as uint8
    (C order)."""
    a = np.ascontiguousarray(a)
    want = {0: np.uint16, 1: np.float32, 2: np.uint8}[dtype]
    if a.dtype != want:
        raise TypeError(f"oracle expects {np.dtype(want).name} for dtype {dtype}, got {a.dtype}")
    return a


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


# ---- closed forms ---------------------------------------------------------------------

def kv_cache_bytes(batch: float, layers: float, tokens: float, hidden: float,
                   bytes_per_value: float) -> float:
    return load().oracle_kv_cache_bytes(batch, layers, tokens, hidden, bytes_per_value)


def topk_count(n: int, p: float) -> int:
    return int(load().oracle_topk_count(n, p))


def num_candidates(L: int, block_size: int, init_tokens: int, local_tokens: int) -> int:
    return int(load().oracle_num_candidates(L, block_size, init_tokens, local_tokens))


# ---- representation vectors ---------------------------------------------------------------

def block_reps(cfg: Mapping, k_cache, page_ids, valid) -> np.ndarray:
    """fp64 mean of each listed page's first ``valid`` keys, per kv head: [n][Hkv][d]."""
    k = _values(k_cache, cfg["dtype"])
    ids, val = _i32(page_ids), _i32(valid)
    n = ids.shape[0]
    out = np.zeros((n, cfg["num_kv_heads"], cfg["head_dim"]), dtype=np.float64)
    c = _cfg(cfg)
    _check(load().oracle_block_reps(ctypes.byref(c), _ptr(k), ctypes.c_int64(k.shape[0]),
                                    _ptr(ids), _ptr(val), ctypes.c_int64(n), _ptr(out)))
    return out


# ---- decode ----------------------------------------------------------------------------------

def _inputs(cfg, q, k_cache, v_cache, block_table, seq_lens, prompt_lens, k_scale=None,
            v_scale=None):
    dt = cfg["dtype"]
    arrs = dict(q=_values(q, 0 if dt == 2 else dt), k=_values(k_cache, dt),
                v=_values(v_cache, dt), bt=_i32(block_table), L=_i32(seq_lens),
                prompt=_i32(seq_lens if prompt_lens is None else prompt_lens))
    if dt == 2:
        shape = arrs["k"].shape[:-1]
        arrs["ks"] = np.ascontiguousarray(k_scale, dtype=np.float32)
        arrs["vs"] = np.ascontiguousarray(v_scale, dtype=np.float32)
        if arrs["ks"].shape != shape or arrs["vs"].shape != shape:
            raise ValueError(f"scales must be {shape}")
    B, max_blocks = arrs["bt"].shape
    ins = _Inputs(_ptr(arrs["q"]), _ptr(arrs["k"]), _ptr(arrs["v"]), arrs["k"].shape[0],
                  _ptr(arrs["bt"]), max_blocks, _ptr(arrs["L"]), _ptr(arrs["prompt"]), B,
                  _ptr(arrs.get("ks")), _ptr(arrs.get("vs")))
    return ins, arrs


def decode(cfg: Mapping, q, k_cache, v_cache, block_table, seq_lens, prompt_lens=None, *,
           units: Sequence[tuple[int, int]] | None = None, sel=None, nsel=None,
           kmax: int | None = None, threads: int = 1, k_scale=None, v_scale=None) -> dict:
    """Decode the listed (request, kv head) units (default: all).

    Returns ``out`` [B][Hq][d] fp64, ``sel`` [B][Hkv][kmax] int32 (ascending block ids,
    -1 padded), ``nsel`` [B][Hkv], ``scores`` [B][Hkv][max_blocks] fp64 (NaN where the
    block is not a candidate).  Rows of units not listed stay zero / -1 / NaN.
    ``sel``/``nsel`` given as inputs replace the oracle's own selection.  With
    ``cfg["dtype"] == 2`` the caches are E4M3 codes with per-row scales ``k_scale`` /
    ``v_scale`` [P][Hkv][S] (R10); pass the selection of the full-precision cache (R11).
    """
    ins, arrs = _inputs(cfg, q, k_cache, v_cache, block_table, seq_lens, prompt_lens,
                        k_scale, v_scale)
    B, max_blocks = arrs["bt"].shape
    Hq, Hkv, d = cfg["num_q_heads"], cfg["num_kv_heads"], cfg["head_dim"]
    if units is None:
        units = [(r, h) for r in range(B) for h in range(Hkv)]
    u = _i32(np.asarray(units, dtype=np.int32).reshape(-1, 2))
    kmax = max_blocks if kmax is None else kmax
    sel_in = None if sel is None else _i32(sel).reshape(B, Hkv, -1)
    if sel_in is not None:
        kmax = max(kmax, sel_in.shape[2])
        pad = np.full((B, Hkv, kmax), -1, np.int32)
        pad[:, :, :sel_in.shape[2]] = sel_in
        sel_in = pad
    nsel_in = None if nsel is None else _i32(nsel).reshape(B, Hkv)
    out = np.zeros((B, Hq, d), np.float64)
    sel_out = np.full((B, Hkv, kmax), -1, np.int32)
    nsel_out = np.zeros((B, Hkv), np.int32)
    scores = np.full((B, Hkv, max_blocks), np.nan, np.float64)
    c = _cfg(cfg)
    _check(load().oracle_decode_units(
        ctypes.byref(c), ctypes.byref(ins), _ptr(u), ctypes.c_int64(u.shape[0]),
        _ptr(sel_in), _ptr(nsel_in), _ptr(sel_out), _ptr(nsel_out), ctypes.c_int32(kmax),
        _ptr(scores), _ptr(out), ctypes.c_int32(threads)))
    return dict(out=out, sel=sel_out, nsel=nsel_out, scores=scores)


# ---- E4M3 compressed pages ---------------------------------------------------------------------

def e4m3_value(codes) -> np.ndarray:
    """fp64 value of each E4M3 code (NaN for S.1111.111)."""
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    out = np.empty(c.shape, np.float64)
    load().oracle_e4m3_values(_ptr(c), ctypes.c_int64(c.size), _ptr(out))
    return out


def e4m3_code(x) -> np.ndarray:
    """R10: nearest E4M3 code of each value (ties to even, saturating at +-448)."""
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty(a.shape, np.uint8)
    load().oracle_e4m3_codes(_ptr(a), ctypes.c_int64(a.size), _ptr(out))
    return out


def quantize_e4m3(cfg: Mapping, cache, page_ids=None) -> tuple[np.ndarray, np.ndarray]:
    """R10 on the listed pages (default: all) of a bf16 cache [P][Hkv][S][d] (uint16 bit
    patterns): (codes [n][Hkv][S][d] uint8, scales [n][Hkv][S] float32)."""
    x = _values(cache, 0)
    ids = _i32(np.arange(x.shape[0]) if page_ids is None else page_ids)
    n = ids.shape[0]
    codes = np.zeros((n,) + x.shape[1:], np.uint8)
    scales = np.zeros((n,) + x.shape[1:3], np.float32)
    c = _cfg(dict(cfg, dtype=0))
    _check(load().oracle_quantize_e4m3(ctypes.byref(c), _ptr(x), ctypes.c_int64(x.shape[0]),
                                       _ptr(ids), ctypes.c_int64(n), _ptr(codes),
                                       _ptr(scales)))
    return codes, scales


def unit_weights(cfg: Mapping, q, k_cache, v_cache, block_table, seq_lens, prompt_lens,
                 r: int, h: int) -> tuple[np.ndarray, np.ndarray]:
    """Softmax weights [G][L] of one unit over every cache position, and its output [G][d]."""
    ins, arrs = _inputs(cfg, q, k_cache, v_cache, block_table, seq_lens, prompt_lens)
    G = cfg["num_q_heads"] // cfg["num_kv_heads"]
    L = int(arrs["L"][r])
    w = np.zeros((G, max(L, 1)), np.float64)
    out = np.zeros((G, cfg["head_dim"]), np.float64)
    c = _cfg(cfg)
    _check(load().oracle_unit(ctypes.byref(c), ctypes.byref(ins), ctypes.c_int32(r),
                              ctypes.c_int32(h), None, ctypes.c_int32(0), None, None,
                              ctypes.c_int32(0), None, _ptr(out), _ptr(w)))
    return w[:, :L], out
