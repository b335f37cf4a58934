"""Python binding of libsrkv (ctypes): the same entry points as ``include/srkv.h``.

Argument marshalling only: every step of the method runs in the library's CUDA
kernels.  Tensors are torch CUDA tensors owned by the caller; streams default to
torch's current stream.  There is no fallback: if ``libsrkv.so`` has not been built
(``python -m block_sparse_retrieval_gb300.build``), :func:`load` raises.

A configuration is a mapping with the keys of :data:`CFG_KEYS` (``dtype`` 0 = bf16,
1 = fp32), e.g. :func:`default_config`.
"""
from __future__ import annotations

import ctypes
import os
from typing import Mapping

import torch

from .build import LIB_PATH

CFG_KEYS = ("num_q_heads", "num_kv_heads", "head_dim", "block_size", "init_tokens",
            "local_tokens", "topk_percent", "dense_boundary", "dtype")
BF16, F32 = 0, 1
EFLAG_PAGE_RANGE, EFLAG_SEQ_LEN, EFLAG_SELECTION, EFLAG_TIMEOUT, EFLAG_PREFIX = 1, 2, 4, 8, 16
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported configuration",
          3: "workspace missing or too small", 4: "CUDA error"}
EXPORTS = ("srkv_default_config", "srkv_status_string", "srkv_topk_count",
           "srkv_num_candidates", "srkv_kmax_bound", "srkv_build_block_reps",
           "srkv_score_topk", "srkv_decode_workspace_size", "srkv_sparse_paged_decode",
           "srkv_retrieval_decode", "srkv_sparse_paged_decode_noalloc",
           "srkv_retrieval_decode_launches", "srkv_append_kv",
           "srkv_retrieval_decode_tiered", "srkv_quantize_kv_fp8",
           "srkv_retrieval_decode_fp8", "srkv_selftest_wait_timeout",
           "srkv_prefix_decode_workspace_size", "srkv_sparse_paged_decode_prefix",
           "srkv_retrieval_decode_prefix", "srkv_host_staging_size",
           "srkv_retrieval_decode_host")
NOALLOC_WORKSPACE_BYTES = 16 << 20


class SrkvError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {STATUS.get(status, status)}")
        self.status = status


class Config(ctypes.Structure):
    _fields_ = [("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("init_tokens", ctypes.c_int32), ("local_tokens", ctypes.c_int32),
                ("topk_percent", ctypes.c_double), ("dense_boundary", ctypes.c_int32),
                ("dtype", ctypes.c_int32)]


_lib: ctypes.CDLL | None = None
_P = ctypes.c_void_p
_I32, _I64, _SZ = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t


def load() -> ctypes.CDLL:
    """Loads the in-tree libsrkv.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: run python -m block_sparse_retrieval_gb300.build")
    lib = ctypes.CDLL(LIB_PATH)
    lib.srkv_default_config.argtypes = [ctypes.POINTER(Config)]
    lib.srkv_default_config.restype = None
    lib.srkv_status_string.argtypes = [ctypes.c_int]
    lib.srkv_status_string.restype = ctypes.c_char_p
    lib.srkv_topk_count.argtypes = [_I64, ctypes.c_double]
    lib.srkv_topk_count.restype = _I64
    lib.srkv_num_candidates.argtypes = [ctypes.POINTER(Config), _I64]
    lib.srkv_num_candidates.restype = _I64
    lib.srkv_kmax_bound.argtypes = [ctypes.POINTER(Config), _I32]
    lib.srkv_kmax_bound.restype = _I32
    lib.srkv_build_block_reps.argtypes = [ctypes.POINTER(Config), _P, _I64, _P, _P, _I32, _P,
                                          _P, _P]
    lib.srkv_append_kv.argtypes = [ctypes.POINTER(Config), _P, _P, _P, _P, _I64, _P, _I32, _P,
                                   _I32, _P, _P, _P]
    lib.srkv_score_topk.argtypes = [ctypes.POINTER(Config), _P, _P, _I64, _P, _I32, _P, _P,
                                    _I32, _P, _I32, _P, _P, _P]
    lib.srkv_decode_workspace_size.argtypes = [ctypes.POINTER(Config), _I32]
    lib.srkv_decode_workspace_size.restype = _SZ
    lib.srkv_retrieval_decode_launches.argtypes = [ctypes.POINTER(Config), _I32, _I32]
    lib.srkv_retrieval_decode_launches.restype = _I32
    lib.srkv_sparse_paged_decode.argtypes = [ctypes.POINTER(Config), _P, _P, _P, _I64, _P, _I32,
                                             _P, _I32, _P, _I32, _P, _P, _P, _SZ, _P, _P]
    lib.srkv_retrieval_decode.argtypes = [ctypes.POINTER(Config), _P, _P, _P, _P, _I64, _P,
                                          _I32, _P, _P, _I32, _P, _I32, _P, _P, _P, _SZ, _P, _P]
    lib.srkv_sparse_paged_decode_noalloc.argtypes = [ctypes.POINTER(Config), _P, _P, _P, _I64,
                                                     _P, _I32, _P, _I32, _P, _I32, _P, _P, _P,
                                                     _P]
    lib.srkv_retrieval_decode_tiered.argtypes = [ctypes.POINTER(Config), _P, _P, _P, _I64, _P,
                                                 _P, _I64, _P, _P, _I32, _P, _P, _I32, _P, _I32,
                                                 _P, _P, _P, _SZ, _P, _P]
    lib.srkv_quantize_kv_fp8.argtypes = [ctypes.POINTER(Config), _P, _P, _I64, _P, _I32, _P, _P,
                                         _P, _P, _P, _P]
    lib.srkv_retrieval_decode_fp8.argtypes = [ctypes.POINTER(Config), _P, _P, _P, _P, _P, _P,
                                              _I64, _P, _I32, _P, _P, _I32, _P, _I32, _P, _P,
                                              _P, _SZ, _P, _P]
    lib.srkv_prefix_decode_workspace_size.argtypes = [ctypes.POINTER(Config), _I32]
    lib.srkv_prefix_decode_workspace_size.restype = _SZ
    lib.srkv_sparse_paged_decode_prefix.argtypes = [ctypes.POINTER(Config), _P, _P, _P, _I64, _P,
                                                    _I32, _P, _I32, _I32, _P, _I32, _P, _P, _P,
                                                    _SZ, _P, _P]
    lib.srkv_retrieval_decode_prefix.argtypes = [ctypes.POINTER(Config), _P, _P, _P, _P, _I64,
                                                 _P, _I32, _P, _P, _I32, _I32, _P, _I32, _P, _P,
                                                 _P, _SZ, _P, _P]
    lib.srkv_host_staging_size.argtypes = [ctypes.POINTER(Config), _I32]
    lib.srkv_host_staging_size.restype = _SZ
    lib.srkv_retrieval_decode_host.argtypes = [ctypes.POINTER(Config), _P, _P, _P, _P, _P, _SZ,
                                               _P, _P, _P, _I64, _P, _I32, _I32, _P, _I32, _P,
                                               _P, _P, _SZ, _P, _P]
    lib.srkv_selftest_wait_timeout.argtypes = [_P, _P]
    lib.srkv_selftest_wait_timeout.restype = ctypes.c_int
    for name in ("srkv_build_block_reps", "srkv_score_topk", "srkv_sparse_paged_decode",
                 "srkv_retrieval_decode", "srkv_sparse_paged_decode_noalloc",
                 "srkv_retrieval_decode_tiered", "srkv_quantize_kv_fp8",
                 "srkv_retrieval_decode_fp8", "srkv_sparse_paged_decode_prefix",
                 "srkv_retrieval_decode_prefix", "srkv_retrieval_decode_host"):
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def config(cfg: Mapping) -> Config:
    return Config(*[cfg[k] for k in CFG_KEYS])


def default_config() -> dict:
    c = Config()
    load().srkv_default_config(ctypes.byref(c))
    return {k: getattr(c, k) for k in CFG_KEYS}


def status_string(status: int) -> str:
    return load().srkv_status_string(status).decode()


def topk_count(n: int, p: float) -> int:
    return int(load().srkv_topk_count(n, p))


def num_candidates(cfg: Mapping, seq_len: int) -> int:
    c = config(cfg)
    return int(load().srkv_num_candidates(ctypes.byref(c), seq_len))


def kmax_bound(cfg: Mapping, max_blocks: int) -> int:
    c = config(cfg)
    return int(load().srkv_kmax_bound(ctypes.byref(c), max_blocks))


def decode_workspace_size(cfg: Mapping, batch: int) -> int:
    c = config(cfg)
    return int(load().srkv_decode_workspace_size(ctypes.byref(c), batch))


def prefix_decode_workspace_size(cfg: Mapping, batch: int) -> int:
    """Workspace bytes of the shared-prefix calls for `batch` requests."""
    c = config(cfg)
    return int(load().srkv_prefix_decode_workspace_size(ctypes.byref(c), batch))


def retrieval_decode_launches(cfg: Mapping, batch: int, max_blocks: int) -> int:
    """Kernels one retrieval_decode call launches on the current device (1 or 3)."""
    c = config(cfg)
    return int(load().srkv_retrieval_decode_launches(ctypes.byref(c), batch, max_blocks))


# ---- marshalling helpers ----------------------------------------------------------------

def _dev(t: torch.Tensor | None, name: str, dtype: torch.dtype | None = None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _host_buf(t: torch.Tensor | None, name: str, dtype: torch.dtype | None = None):
    """A host tensor (page-locked or not) as a pointer."""
    if t is None:
        return None
    if t.is_cuda:
        raise ValueError(f"{name} must be a host tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _store_dtype(cfg: Mapping) -> torch.dtype:
    return torch.bfloat16 if cfg["dtype"] == BF16 else torch.float32


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        if _raw_stream is not None:  # the current stream's handle, without a Stream object
            return ctypes.c_void_p(_raw_stream(torch.cuda.current_device()))
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(status: int, where: str) -> None:
    if status != 0:
        raise SrkvError(status, where)


def _shape(t: torch.Tensor | None, name: str, *dims) -> None:
    """t (if given) has len(dims) dimensions of those sizes; None matches any size.  The
    library sees only pointers, so a tensor of the wrong shape would be read or written out
    of its bounds: the shapes are checked here, before anything is launched."""
    if t is None:
        return
    s = t.shape
    if len(s) == len(dims):
        for g, w in zip(s, dims):
            if w is not None and g != w:
                break
        else:
            return
    want = "[" + ", ".join("*" if w is None else str(w) for w in dims) + "]"
    raise ValueError(f"{name} must have shape {want}, got {list(s)}")


def _rows(t: torch.Tensor, name: str, at_least: int) -> None:
    if t.shape[0] < at_least:
        raise ValueError(f"{name} needs at least {at_least} rows, got {t.shape[0]}")


def _cache_dims(cfg: Mapping) -> tuple[int, int, int, int]:
    return cfg["num_q_heads"], cfg["num_kv_heads"], cfg["block_size"], cfg["head_dim"]


def _step_shapes(cfg: Mapping, q, k_cache, v_cache, block_table, seq_lens, prompt_lens, sel,
                 nsel, out, reps=None, reps_rows: int = 0) -> tuple[int, int]:
    """Shapes shared by the decode entry points; returns (batch, max_blocks)."""
    Hq, Hkv, S, d = _cache_dims(cfg)
    _shape(block_table, "block_table", None, None)
    B, max_blocks = block_table.shape
    _shape(q, "q", B, Hq, d)
    _shape(k_cache, "k_cache", None, Hkv, S, d)
    _shape(v_cache, "v_cache", k_cache.shape[0], Hkv, S, d)
    _shape(seq_lens, "seq_lens", B)
    _shape(prompt_lens, "prompt_lens", B)
    _shape(sel, "sel", B, Hkv, None)
    _shape(nsel, "nsel", B, Hkv)
    _shape(out, "out", B, Hq, d)
    if reps is not None:
        _shape(reps, "reps", None, Hkv, d)
        _rows(reps, "reps", reps_rows)
    return B, max_blocks


# ---- entry points --------------------------------------------------------------------------

def build_block_reps(cfg: Mapping, k_cache: torch.Tensor, page_ids: torch.Tensor,
                     page_valid_tokens: torch.Tensor, reps: torch.Tensor,
                     error_flags: torch.Tensor | None = None, stream=None) -> None:
    _, Hkv, S, d = _cache_dims(cfg)
    _shape(k_cache, "k_cache", None, Hkv, S, d)
    _shape(page_ids, "page_ids", None)
    _shape(page_valid_tokens, "page_valid_tokens", page_ids.numel())
    _shape(reps, "reps", None, Hkv, d)
    _rows(reps, "reps", k_cache.shape[0])
    c = config(cfg)
    _check(load().srkv_build_block_reps(
        ctypes.byref(c), _dev(k_cache, "k_cache", _store_dtype(cfg)), k_cache.shape[0],
        _dev(page_ids, "page_ids", torch.int32), _dev(page_valid_tokens, "page_valid_tokens",
                                                      torch.int32),
        page_ids.numel(), _dev(reps, "reps", torch.float32),
        _dev(error_flags, "error_flags", torch.int32), _stream(stream)), "srkv_build_block_reps")


def append_kv(cfg: Mapping, k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
              v_cache: torch.Tensor, block_table: torch.Tensor, seq_lens: torch.Tensor,
              reps: torch.Tensor, error_flags: torch.Tensor | None = None,
              stream=None) -> None:
    """Writes each request's new token (k_new, v_new: [B][Hkv][d]) at position seq_lens[r]
    and refreshes that page's representation vector; the caller then advances seq_lens."""
    _, Hkv, S, d = _cache_dims(cfg)
    _shape(block_table, "block_table", None, None)
    B = block_table.shape[0]
    _shape(k_new, "k_new", B, Hkv, d)
    _shape(v_new, "v_new", B, Hkv, d)
    _shape(k_cache, "k_cache", None, Hkv, S, d)
    _shape(v_cache, "v_cache", k_cache.shape[0], Hkv, S, d)
    _shape(seq_lens, "seq_lens", B)
    _shape(reps, "reps", None, Hkv, d)
    _rows(reps, "reps", k_cache.shape[0])
    c = config(cfg)
    st = _store_dtype(cfg)
    _check(load().srkv_append_kv(
        ctypes.byref(c), _dev(k_new, "k_new", st), _dev(v_new, "v_new", st),
        _dev(k_cache, "k_cache", st), _dev(v_cache, "v_cache", st), k_cache.shape[0],
        _dev(block_table, "block_table", torch.int32), block_table.shape[1],
        _dev(seq_lens, "seq_lens", torch.int32), seq_lens.numel(),
        _dev(reps, "reps", torch.float32), _dev(error_flags, "error_flags", torch.int32),
        _stream(stream)), "srkv_append_kv")


def score_topk(cfg: Mapping, q: torch.Tensor, reps: torch.Tensor, block_table: torch.Tensor,
               seq_lens: torch.Tensor, prompt_lens: torch.Tensor | None, sel: torch.Tensor,
               nsel: torch.Tensor, error_flags: torch.Tensor | None = None,
               stream=None) -> None:
    Hq, Hkv, _, d = _cache_dims(cfg)
    _shape(block_table, "block_table", None, None)
    B, max_blocks = block_table.shape
    _shape(q, "q", B, Hq, d)
    _shape(reps, "reps", None, Hkv, d)
    _shape(seq_lens, "seq_lens", B)
    _shape(prompt_lens, "prompt_lens", B)
    _shape(sel, "sel", B, Hkv, None)
    _shape(nsel, "nsel", B, Hkv)
    c = config(cfg)
    _check(load().srkv_score_topk(
        ctypes.byref(c), _dev(q, "q", _store_dtype(cfg)), _dev(reps, "reps", torch.float32),
        reps.shape[0], _dev(block_table, "block_table", torch.int32), max_blocks,
        _dev(seq_lens, "seq_lens", torch.int32), _dev(prompt_lens, "prompt_lens", torch.int32),
        B, _dev(sel, "sel", torch.int32), sel.shape[-1], _dev(nsel, "nsel", torch.int32),
        _dev(error_flags, "error_flags", torch.int32), _stream(stream)), "srkv_score_topk")


def sparse_paged_decode(cfg: Mapping, q: torch.Tensor, k_cache: torch.Tensor,
                        v_cache: torch.Tensor, block_table: torch.Tensor,
                        seq_lens: torch.Tensor, sel: torch.Tensor, nsel: torch.Tensor,
                        out: torch.Tensor, workspace: torch.Tensor,
                        error_flags: torch.Tensor | None = None, stream=None) -> None:
    B, max_blocks = _step_shapes(cfg, q, k_cache, v_cache, block_table, seq_lens, None, sel,
                                 nsel, out)
    c = config(cfg)
    dt = _store_dtype(cfg)
    _check(load().srkv_sparse_paged_decode(
        ctypes.byref(c), _dev(q, "q", dt), _dev(k_cache, "k_cache", dt),
        _dev(v_cache, "v_cache", dt), k_cache.shape[0],
        _dev(block_table, "block_table", torch.int32), max_blocks,
        _dev(seq_lens, "seq_lens", torch.int32), B, _dev(sel, "sel", torch.int32),
        sel.shape[-1], _dev(nsel, "nsel", torch.int32), _dev(out, "out", dt),
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _dev(error_flags, "error_flags", torch.int32), _stream(stream)),
        "srkv_sparse_paged_decode")


def retrieval_decode(cfg: Mapping, q: torch.Tensor, k_cache: torch.Tensor,
                     v_cache: torch.Tensor, reps: torch.Tensor, block_table: torch.Tensor,
                     seq_lens: torch.Tensor, prompt_lens: torch.Tensor | None,
                     sel: torch.Tensor, nsel: torch.Tensor, out: torch.Tensor,
                     workspace: torch.Tensor, error_flags: torch.Tensor | None = None,
                     stream=None) -> None:
    B, max_blocks = _step_shapes(cfg, q, k_cache, v_cache, block_table, seq_lens, prompt_lens,
                                 sel, nsel, out, reps, k_cache.shape[0])
    c = config(cfg)
    dt = _store_dtype(cfg)
    _check(load().srkv_retrieval_decode(
        ctypes.byref(c), _dev(q, "q", dt), _dev(k_cache, "k_cache", dt),
        _dev(v_cache, "v_cache", dt), _dev(reps, "reps", torch.float32), k_cache.shape[0],
        _dev(block_table, "block_table", torch.int32), max_blocks,
        _dev(seq_lens, "seq_lens", torch.int32), _dev(prompt_lens, "prompt_lens", torch.int32),
        B, _dev(sel, "sel", torch.int32), sel.shape[-1], _dev(nsel, "nsel", torch.int32),
        _dev(out, "out", dt), _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(),
        _dev(error_flags, "error_flags", torch.int32), _stream(stream)), "srkv_retrieval_decode")


def host_staging_size(cfg: Mapping, batch: int) -> int:
    """Bytes of device staging srkv_retrieval_decode_host needs for `batch` requests."""
    c = config(cfg)
    return int(load().srkv_host_staging_size(ctypes.byref(c), batch))


def host_inputs(cfg: Mapping, batch: int) -> dict:
    """Page-locked host tensors for srkv_retrieval_decode_host laid out like its staging (q,
    then seq_lens, then prompt_lens, each at a 256-byte boundary, in one buffer), so that the
    call copies them in one go: {"q": [batch][Hq][d], "seq_lens": [batch], "prompt_lens":
    [batch]} (views of one buffer)."""
    Hq, _, _, d = _cache_dims(cfg)
    dt = _store_dtype(cfg)
    qb = batch * Hq * d * (2 if dt == torch.bfloat16 else 4)
    r256 = lambda x: (x + 255) // 256 * 256
    buf = torch.zeros(host_staging_size(cfg, batch), dtype=torch.uint8).pin_memory()
    lo = r256(qb)
    return {"q": buf[:qb].view(dt).view(batch, Hq, d),
            "seq_lens": buf[lo:lo + 4 * batch].view(torch.int32),
            "prompt_lens": buf[lo + r256(4 * batch):lo + r256(4 * batch) + 4 * batch].view(
                torch.int32)}


def retrieval_decode_host(cfg: Mapping, q_host: torch.Tensor, seq_lens_host: torch.Tensor,
                          prompt_lens_host: torch.Tensor | None, out_host: torch.Tensor,
                          staging: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                          reps: torch.Tensor, block_table: torch.Tensor, sel: torch.Tensor,
                          nsel: torch.Tensor, out: torch.Tensor, workspace: torch.Tensor,
                          error_flags: torch.Tensor | None = None, stream=None) -> None:
    """srkv_retrieval_decode_host: the query and lengths from host tensors (page-locked for
    asynchronous copies), the output into a host tensor; returns once out_host holds it."""
    B, max_blocks = _step_shapes(cfg, q_host, k_cache, v_cache, block_table, seq_lens_host,
                                 prompt_lens_host, sel, nsel, out, reps, k_cache.shape[0])
    _shape(out_host, "out_host", *out.shape)
    c = config(cfg)
    dt = _store_dtype(cfg)
    _check(load().srkv_retrieval_decode_host(
        ctypes.byref(c), _host_buf(q_host, "q_host", dt),
        _host_buf(seq_lens_host, "seq_lens_host", torch.int32),
        _host_buf(prompt_lens_host, "prompt_lens_host", torch.int32),
        _host_buf(out_host, "out_host", dt), _dev(staging, "staging"),
        staging.numel() * staging.element_size(), _dev(k_cache, "k_cache", dt),
        _dev(v_cache, "v_cache", dt), _dev(reps, "reps", torch.float32), k_cache.shape[0],
        _dev(block_table, "block_table", torch.int32), max_blocks, B,
        _dev(sel, "sel", torch.int32), sel.shape[-1], _dev(nsel, "nsel", torch.int32),
        _dev(out, "out", dt), _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(),
        _dev(error_flags, "error_flags", torch.int32), _stream(stream)),
        "srkv_retrieval_decode_host")


class HostDecodeStep:
    """srkv_retrieval_decode_host over fixed buffers (a serving loop's): the arguments are
    checked and marshalled once, here; each call runs one step with the buffers' current
    contents and returns once out_host holds the output."""

    def __init__(self, cfg: Mapping, q_host: torch.Tensor, seq_lens_host: torch.Tensor,
                 prompt_lens_host: torch.Tensor | None, out_host: torch.Tensor,
                 staging: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                 reps: torch.Tensor, block_table: torch.Tensor, sel: torch.Tensor,
                 nsel: torch.Tensor, out: torch.Tensor, workspace: torch.Tensor,
                 error_flags: torch.Tensor | None = None, stream=None):
        B, max_blocks = _step_shapes(cfg, q_host, k_cache, v_cache, block_table, seq_lens_host,
                                     prompt_lens_host, sel, nsel, out, reps, k_cache.shape[0])
        _shape(out_host, "out_host", *out.shape)
        dt = _store_dtype(cfg)
        self._cfg = config(cfg)
        # the tensors stay referenced as long as the step: their memory is what it reads
        self._keep = (q_host, seq_lens_host, prompt_lens_host, out_host, staging, k_cache,
                      v_cache, reps, block_table, sel, nsel, out, workspace, error_flags)
        self._fn = load().srkv_retrieval_decode_host
        self._args = (
            ctypes.byref(self._cfg), _host_buf(q_host, "q_host", dt),
            _host_buf(seq_lens_host, "seq_lens_host", torch.int32),
            _host_buf(prompt_lens_host, "prompt_lens_host", torch.int32),
            _host_buf(out_host, "out_host", dt), _dev(staging, "staging"),
            staging.numel() * staging.element_size(), _dev(k_cache, "k_cache", dt),
            _dev(v_cache, "v_cache", dt), _dev(reps, "reps", torch.float32), k_cache.shape[0],
            _dev(block_table, "block_table", torch.int32), max_blocks, B,
            _dev(sel, "sel", torch.int32), sel.shape[-1], _dev(nsel, "nsel", torch.int32),
            _dev(out, "out", dt), _dev(workspace, "workspace"),
            workspace.numel() * workspace.element_size(),
            _dev(error_flags, "error_flags", torch.int32), _stream(stream))

    def __call__(self) -> None:
        _check(self._fn(*self._args), "srkv_retrieval_decode_host")


def sparse_paged_decode_prefix(cfg: Mapping, q: torch.Tensor, k_cache: torch.Tensor,
                               v_cache: torch.Tensor, block_table: torch.Tensor,
                               seq_lens: torch.Tensor, prefix_blocks: int, sel: torch.Tensor,
                               nsel: torch.Tensor, out: torch.Tensor, workspace: torch.Tensor,
                               error_flags: torch.Tensor | None = None, stream=None) -> None:
    """srkv_sparse_paged_decode_prefix: the first prefix_blocks logical blocks of every request
    are the same pages, attended once per kv head for all requests."""
    B, max_blocks = _step_shapes(cfg, q, k_cache, v_cache, block_table, seq_lens, None, sel,
                                 nsel, out)
    c = config(cfg)
    dt = _store_dtype(cfg)
    _check(load().srkv_sparse_paged_decode_prefix(
        ctypes.byref(c), _dev(q, "q", dt), _dev(k_cache, "k_cache", dt),
        _dev(v_cache, "v_cache", dt), k_cache.shape[0],
        _dev(block_table, "block_table", torch.int32), max_blocks,
        _dev(seq_lens, "seq_lens", torch.int32), B, prefix_blocks,
        _dev(sel, "sel", torch.int32), sel.shape[-1], _dev(nsel, "nsel", torch.int32),
        _dev(out, "out", dt), _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(),
        _dev(error_flags, "error_flags", torch.int32), _stream(stream)),
        "srkv_sparse_paged_decode_prefix")


def retrieval_decode_prefix(cfg: Mapping, q: torch.Tensor, k_cache: torch.Tensor,
                            v_cache: torch.Tensor, reps: torch.Tensor, block_table: torch.Tensor,
                            seq_lens: torch.Tensor, prompt_lens: torch.Tensor | None,
                            prefix_blocks: int, sel: torch.Tensor, nsel: torch.Tensor,
                            out: torch.Tensor, workspace: torch.Tensor,
                            error_flags: torch.Tensor | None = None, stream=None) -> None:
    """srkv_retrieval_decode_prefix: scoring and selection, then the decode with the shared
    prefix attended once per kv head for all requests."""
    B, max_blocks = _step_shapes(cfg, q, k_cache, v_cache, block_table, seq_lens, prompt_lens,
                                 sel, nsel, out, reps, k_cache.shape[0])
    c = config(cfg)
    dt = _store_dtype(cfg)
    _check(load().srkv_retrieval_decode_prefix(
        ctypes.byref(c), _dev(q, "q", dt), _dev(k_cache, "k_cache", dt),
        _dev(v_cache, "v_cache", dt), _dev(reps, "reps", torch.float32), k_cache.shape[0],
        _dev(block_table, "block_table", torch.int32), max_blocks,
        _dev(seq_lens, "seq_lens", torch.int32), _dev(prompt_lens, "prompt_lens", torch.int32),
        B, prefix_blocks, _dev(sel, "sel", torch.int32), sel.shape[-1],
        _dev(nsel, "nsel", torch.int32), _dev(out, "out", dt), _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(),
        _dev(error_flags, "error_flags", torch.int32), _stream(stream)),
        "srkv_retrieval_decode_prefix")


def _host(t: torch.Tensor | None, name: str, dtype: torch.dtype):
    if t is None:
        return None
    if t.is_cuda or not t.is_pinned():
        raise ValueError(f"{name} must be a pinned host tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def retrieval_decode_tiered(cfg: Mapping, q: torch.Tensor, k_cache: torch.Tensor,
                            v_cache: torch.Tensor, k_host: torch.Tensor | None,
                            v_host: torch.Tensor | None, reps: torch.Tensor,
                            block_table: torch.Tensor, seq_lens: torch.Tensor,
                            prompt_lens: torch.Tensor | None, sel: torch.Tensor,
                            nsel: torch.Tensor, out: torch.Tensor, workspace: torch.Tensor,
                            error_flags: torch.Tensor | None = None, stream=None) -> None:
    """srkv_retrieval_decode_tiered: page ids >= k_cache.shape[0] name pages of the pinned
    host pool k_host / v_host (page id - k_cache.shape[0])."""
    _, Hkv, S, d = _cache_dims(cfg)
    n_host = 0 if k_host is None else k_host.shape[0]
    _shape(k_host, "k_host", None, Hkv, S, d)
    _shape(v_host, "v_host", n_host, Hkv, S, d)
    B, max_blocks = _step_shapes(cfg, q, k_cache, v_cache, block_table, seq_lens, prompt_lens,
                                 sel, nsel, out, reps, k_cache.shape[0] + n_host)
    c = config(cfg)
    dt = _store_dtype(cfg)
    _check(load().srkv_retrieval_decode_tiered(
        ctypes.byref(c), _dev(q, "q", dt), _dev(k_cache, "k_cache", dt),
        _dev(v_cache, "v_cache", dt), k_cache.shape[0], _host(k_host, "k_host", dt),
        _host(v_host, "v_host", dt), n_host, _dev(reps, "reps", torch.float32),
        _dev(block_table, "block_table", torch.int32), max_blocks,
        _dev(seq_lens, "seq_lens", torch.int32), _dev(prompt_lens, "prompt_lens", torch.int32),
        B, _dev(sel, "sel", torch.int32), sel.shape[-1], _dev(nsel, "nsel", torch.int32),
        _dev(out, "out", dt), _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(),
        _dev(error_flags, "error_flags", torch.int32), _stream(stream)),
        "srkv_retrieval_decode_tiered")


def quantize_kv_fp8(cfg: Mapping, k_cache: torch.Tensor, v_cache: torch.Tensor,
                    page_ids: torch.Tensor, k_fp8: torch.Tensor, v_fp8: torch.Tensor,
                    k_scale: torch.Tensor, v_scale: torch.Tensor,
                    error_flags: torch.Tensor | None = None, stream=None) -> None:
    """srkv_quantize_kv_fp8: pages page_ids of the bf16 caches as E4M3 codes (uint8 tensors
    of the caches' shape) with one fp32 scale per (page, kv head, token) row."""
    _, Hkv, S, d = _cache_dims(cfg)
    _shape(k_cache, "k_cache", None, Hkv, S, d)
    P = k_cache.shape[0]
    _shape(v_cache, "v_cache", P, Hkv, S, d)
    _shape(page_ids, "page_ids", None)
    for t, name in ((k_fp8, "k_fp8"), (v_fp8, "v_fp8")):
        _shape(t, name, P, Hkv, S, d)
    for t, name in ((k_scale, "k_scale"), (v_scale, "v_scale")):
        _shape(t, name, P, Hkv, S)
    c = config(cfg)
    _check(load().srkv_quantize_kv_fp8(
        ctypes.byref(c), _dev(k_cache, "k_cache", torch.bfloat16),
        _dev(v_cache, "v_cache", torch.bfloat16), k_cache.shape[0],
        _dev(page_ids, "page_ids", torch.int32), page_ids.numel(),
        _dev(k_fp8, "k_fp8", torch.uint8), _dev(v_fp8, "v_fp8", torch.uint8),
        _dev(k_scale, "k_scale", torch.float32), _dev(v_scale, "v_scale", torch.float32),
        _dev(error_flags, "error_flags", torch.int32), _stream(stream)), "srkv_quantize_kv_fp8")


def retrieval_decode_fp8(cfg: Mapping, q: torch.Tensor, k_fp8: torch.Tensor,
                         v_fp8: torch.Tensor, k_scale: torch.Tensor, v_scale: torch.Tensor,
                         reps: torch.Tensor, block_table: torch.Tensor, seq_lens: torch.Tensor,
                         prompt_lens: torch.Tensor | None, sel: torch.Tensor, nsel: torch.Tensor,
                         out: torch.Tensor, workspace: torch.Tensor,
                         error_flags: torch.Tensor | None = None, stream=None) -> None:
    """srkv_retrieval_decode_fp8: the decode step over E4M3 pages (bf16 query and output)."""
    _, Hkv, S, _ = _cache_dims(cfg)
    B, max_blocks = _step_shapes(cfg, q, k_fp8, v_fp8, block_table, seq_lens, prompt_lens,
                                 sel, nsel, out, reps, k_fp8.shape[0])
    for t, name in ((k_scale, "k_scale"), (v_scale, "v_scale")):
        _shape(t, name, k_fp8.shape[0], Hkv, S)
    c = config(cfg)
    _check(load().srkv_retrieval_decode_fp8(
        ctypes.byref(c), _dev(q, "q", torch.bfloat16), _dev(k_fp8, "k_fp8", torch.uint8),
        _dev(v_fp8, "v_fp8", torch.uint8), _dev(k_scale, "k_scale", torch.float32),
        _dev(v_scale, "v_scale", torch.float32), _dev(reps, "reps", torch.float32),
        k_fp8.shape[0], _dev(block_table, "block_table", torch.int32), max_blocks,
        _dev(seq_lens, "seq_lens", torch.int32), _dev(prompt_lens, "prompt_lens", torch.int32),
        B, _dev(sel, "sel", torch.int32), sel.shape[-1], _dev(nsel, "nsel", torch.int32),
        _dev(out, "out", torch.bfloat16), _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(),
        _dev(error_flags, "error_flags", torch.int32), _stream(stream)),
        "srkv_retrieval_decode_fp8")


def selftest_wait_timeout(error_flags: torch.Tensor, stream=None) -> None:
    """srkv_selftest_wait_timeout: a kernel whose bounded waits never see an arrival; they
    give up after their limit and set SRKV_EFLAG_TIMEOUT in error_flags."""
    _check(load().srkv_selftest_wait_timeout(_dev(error_flags, "error_flags", torch.int32),
                                             _stream(stream)), "srkv_selftest_wait_timeout")


def sparse_paged_decode_noalloc(cfg: Mapping, q: torch.Tensor, k_cache: torch.Tensor,
                                v_cache: torch.Tensor, block_table: torch.Tensor,
                                seq_lens: torch.Tensor, sel: torch.Tensor, nsel: torch.Tensor,
                                out: torch.Tensor, error_flags: torch.Tensor | None = None,
                                stream=None) -> None:
    """srkv_sparse_paged_decode with the library's own static scratch (no workspace)."""
    B, max_blocks = _step_shapes(cfg, q, k_cache, v_cache, block_table, seq_lens, None, sel,
                                 nsel, out)
    c = config(cfg)
    dt = _store_dtype(cfg)
    _check(load().srkv_sparse_paged_decode_noalloc(
        ctypes.byref(c), _dev(q, "q", dt), _dev(k_cache, "k_cache", dt),
        _dev(v_cache, "v_cache", dt), k_cache.shape[0],
        _dev(block_table, "block_table", torch.int32), max_blocks,
        _dev(seq_lens, "seq_lens", torch.int32), B, _dev(sel, "sel", torch.int32),
        sel.shape[-1], _dev(nsel, "nsel", torch.int32), _dev(out, "out", dt),
        _dev(error_flags, "error_flags", torch.int32), _stream(stream)),
        "srkv_sparse_paged_decode_noalloc")


# ---- buffers for a step --------------------------------------------------------------------

class DecodeBuffers:
    """Device buffers one decode step needs besides the cache: reps, selection, output,
    workspace and the error word.  Allocated once by torch (the library allocates none)."""

    def __init__(self, cfg: Mapping, batch: int, max_blocks: int, num_pages: int,
                 device="cuda", prefix: bool = False):
        Hq, Hkv, d = cfg["num_q_heads"], cfg["num_kv_heads"], cfg["head_dim"]
        self.kmax = max(1, kmax_bound(cfg, max_blocks))
        self.reps = torch.zeros(num_pages, Hkv, d, dtype=torch.float32, device=device)
        self.sel = torch.full((batch, Hkv, self.kmax), -1, dtype=torch.int32, device=device)
        self.nsel = torch.zeros(batch, Hkv, dtype=torch.int32, device=device)
        self.out = torch.zeros(batch, Hq, d, dtype=_store_dtype(cfg), device=device)
        # prefix: sized for the shared-prefix calls too
        nbytes = (prefix_decode_workspace_size if prefix else decode_workspace_size)(cfg, batch)
        self.workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        self.error_flags = torch.zeros(1, dtype=torch.int32, device=device)
