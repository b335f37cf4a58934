"""The C ABI on the host (no GPU needed): the library builds and loads, exports every
function include/srkv.h declares, and its host-side helpers and argument checks behave.
None of these calls reaches a kernel launch."""
import ctypes
import os
import re

import pytest

import oracle
from block_sparse_retrieval_gb300 import build, srkv

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "srkv.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return srkv.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(srkv_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert set(declared_functions()) == set(srkv.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_defaults_are_the_pages_knobs(lib):
    cfg = srkv.default_config()
    assert (cfg["init_tokens"], cfg["local_tokens"], cfg["block_size"]) == (1024, 7192, 128)
    assert cfg["topk_percent"] == 0.2 and cfg["dense_boundary"] == 32768


def test_topk_count_matches_the_oracle(lib):
    for p in [i / 100 for i in range(0, 101)] + [1 / 3]:
        for n in range(0, 1500):
            assert srkv.topk_count(n, p) == oracle.topk_count(n, p), (n, p)


def test_num_candidates_matches_the_oracle(lib):
    cfg = srkv.default_config()
    for init in (0, 100, 1024, 1000):
        for local in (0, 7192, 1024, 50):
            c = dict(cfg, init_tokens=init, local_tokens=local)
            for L in list(range(0, 3000, 37)) + [65536, 131072, 131071, 8216, 8217]:
                assert srkv.num_candidates(c, L) == oracle.num_candidates(L, 128, init, local)


def test_kmax_bound(lib):
    cfg = srkv.default_config()
    # dense mode possible -> every candidate of a max-length request
    assert srkv.kmax_bound(cfg, 1024) == oracle.num_candidates(1024 * 128, 128, 1024, 7192)
    sparse = dict(cfg, dense_boundary=0)
    assert srkv.kmax_bound(sparse, 1024) == oracle.topk_count(960, 0.2) == 192


def test_status_strings(lib):
    for s in range(5):
        assert srkv.status_string(s) == srkv.STATUS[s]
    assert srkv.status_string(99) == "unknown status"


def test_workspace_size_is_device_independent_and_grows(lib):
    cfg = srkv.default_config()
    a, b = srkv.decode_workspace_size(cfg, 1), srkv.decode_workspace_size(cfg, 64)
    assert 0 < a < b and a % 256 == 0
    assert srkv.decode_workspace_size(dict(cfg, head_dim=96), 1) == 0


def _call_decode(lib, cfg, **over):
    c = srkv.config(cfg)
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the checks reject the call first
    args = dict(q=fake, k=fake, v=fake, num_pages=10, bt=fake, max_blocks=8, seq=fake, batch=1,
                sel=fake, kmax=8, nsel=fake, out=fake, ws=None, ws_bytes=0, flags=None)
    args.update(over)
    return lib.srkv_sparse_paged_decode(
        ctypes.byref(c), args["q"], args["k"], args["v"], args["num_pages"], args["bt"],
        args["max_blocks"], args["seq"], args["batch"], args["sel"], args["kmax"], args["nsel"],
        args["out"], args["ws"], args["ws_bytes"], args["flags"], None)


def test_decode_argument_checks(lib):
    cfg = srkv.default_config()
    assert _call_decode(lib, cfg, q=None) == 1
    assert _call_decode(lib, cfg, k=ctypes.c_void_p((1 << 20) + 8)) == 1   # misaligned
    assert _call_decode(lib, dict(cfg, block_size=64)) == 1
    assert _call_decode(lib, dict(cfg, num_q_heads=30)) == 1
    assert _call_decode(lib, dict(cfg, topk_percent=1.5)) == 1
    assert _call_decode(lib, dict(cfg, head_dim=80)) == 1
    assert _call_decode(lib, cfg, max_blocks=0) == 1
    assert _call_decode(lib, cfg) == 3                                      # no workspace
    assert _call_decode(lib, cfg, ws=ctypes.c_void_p(1 << 20), ws_bytes=16) == 3
    assert _call_decode(lib, cfg, batch=0) == 0                             # nothing to do
    # bf16 groups above 16 heads have no kernel
    assert _call_decode(lib, dict(cfg, dtype=1, num_q_heads=8 * 17)) == 2


def test_prefix_argument_checks(lib):
    cfg = srkv.default_config()
    c = srkv.config(cfg)
    fake = ctypes.c_void_p(1 << 20)

    def call(cfg_, prefix, max_blocks=8, ws=None, ws_bytes=0):
        cc = srkv.config(cfg_)
        return lib.srkv_sparse_paged_decode_prefix(
            ctypes.byref(cc), fake, fake, fake, 10, fake, max_blocks, fake, 1, prefix, fake, 8,
            fake, fake, ws, ws_bytes, None, None)
    assert call(cfg, -1) == 1
    assert call(cfg, 9) == 1                                    # longer than the block table
    assert call(dict(cfg, head_dim=64), 2) == 2                 # the cascade takes d 128
    assert call(dict(cfg, num_q_heads=8 * 3), 2) == 2           # group 3
    assert call(cfg, 2049, max_blocks=4096) == 2                # at most 2048 shared blocks
    assert call(cfg, 2) == 3                                    # no workspace
    small = srkv.decode_workspace_size(cfg, 1)
    assert srkv.prefix_decode_workspace_size(cfg, 1) > small
    assert call(cfg, 2, ws=fake, ws_bytes=small) == 3           # the plain call's is too small
    assert lib.srkv_retrieval_decode_prefix(ctypes.byref(c), fake, fake, fake, fake, 10, fake, 8,
                                            fake, None, 1, -1, fake, 8, fake, fake, None, 0,
                                            None, None) == 1


def test_host_call_staging_and_argument_checks(lib):
    cfg = srkv.default_config()
    c = srkv.config(cfg)
    # q (batch x 32 heads x 128 x 2 bytes), then the lengths and the prompt lengths, each at a
    # 256-byte boundary
    assert srkv.host_staging_size(cfg, 1) == 8192 + 256 + 256
    assert srkv.host_staging_size(cfg, 3) == 24576 + 256 + 256
    assert srkv.host_staging_size(dict(cfg, dtype=1), 1) == 16384 + 512
    assert lib.srkv_host_staging_size(None, 1) == 0
    fake = ctypes.c_void_p(1 << 20)
    host = ctypes.c_void_p(1 << 21)

    def call(q=host, lens=host, out_host=host, staging=fake, staging_bytes=1 << 16, batch=1):
        return lib.srkv_retrieval_decode_host(
            ctypes.byref(c), q, lens, None, out_host, staging, staging_bytes, fake, fake, fake,
            10, fake, 8, batch, fake, 8, fake, fake, None, 0, None, None)
    # rejected before any copy or launch
    assert call(q=None) == 1
    assert call(lens=None) == 1
    assert call(out_host=None) == 1
    assert call(staging=None) == 1
    assert call(staging_bytes=8192) == 1                        # smaller than the staging size
    assert call(staging=ctypes.c_void_p((1 << 20) + 16)) == 1   # not 256-byte aligned
    assert call(batch=-1) == 1


def test_score_topk_argument_checks(lib):
    cfg = dict(srkv.default_config(), dense_boundary=0)
    c = srkv.config(cfg)
    fake = ctypes.c_void_p(1 << 20)
    call = lambda kmax, q=fake: lib.srkv_score_topk(ctypes.byref(c), q, fake, 10, fake, 1024,
                                                    fake, None, 1, fake, kmax, fake, None, None)
    assert call(191) == 1                    # below srkv_kmax_bound (192)
    assert call(192, q=None) == 1
    assert call(-1) == 1
    # keys and pages of every candidate stay on chip: 25 600 blocks at most
    wide = lambda mb: lib.srkv_score_topk(ctypes.byref(c), fake, fake, 10, fake, mb, fake,
                                          None, 1, fake, 1 << 20, fake, None, None)
    assert wide(25601) == 2


def test_build_reps_argument_checks(lib):
    cfg = srkv.default_config()
    c = srkv.config(cfg)
    fake = ctypes.c_void_p(1 << 20)
    assert lib.srkv_build_block_reps(ctypes.byref(c), fake, 10, fake, fake, 0, fake, None,
                                     None) == 0
    assert lib.srkv_build_block_reps(ctypes.byref(c), None, 10, fake, fake, 3, fake, None,
                                     None) == 1
    assert lib.srkv_build_block_reps(None, fake, 10, fake, fake, 3, fake, None, None) == 1
