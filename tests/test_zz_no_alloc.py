"""The decode entry point that needs no workspace from its caller.

srkv_sparse_paged_decode_noalloc serves callers that cannot allocate device memory on their
decode path (code under CUDA-graph stream capture, serving loops that forbid allocator
calls, plugins handed only their input and output buffers): its scratch is a static device
array inside the library.  These checks call it through the C ABI and compare it with the
workspace-taking entry point.  Both run the same split kernel and combine with the same plan
and grid, so their outputs must be equal to the bit.  Calls alternate between a larger and a
smaller batch, so a call that read a value the previous call left in the shared array, rather
than one it wrote itself, would show; the workspace path runs on a workspace filled with
0xFF bytes (NaN as fp32), so it too reads nothing it did not write.
"""
import ctypes

import pytest
import torch

from block_sparse_retrieval_gb300 import srkv, synth
from parity import gpu_select

pytestmark = pytest.mark.gpu


def _noalloc(lib, case, sel, nsel, out, flags):
    c = srkv.config(case.cfg)
    B, max_blocks = case.block_table.shape
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    return lib.srkv_sparse_paged_decode_noalloc(
        ctypes.byref(c), p(case.q), p(case.k_cache), p(case.v_cache), case.k_cache.shape[0],
        p(case.block_table), max_blocks, p(case.seq_lens), B, p(sel), sel.shape[-1], p(nsel),
        p(out), p(flags), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _workspace_out(case, buf):
    """srkv_sparse_paged_decode on a workspace whose every byte is 0xFF."""
    buf.workspace.fill_(0xFF)
    buf.error_flags.zero_()
    out = torch.full_like(buf.out, float("nan"))
    srkv.sparse_paged_decode(case.cfg, case.q, case.k_cache, case.v_cache, case.block_table,
                             case.seq_lens, buf.sel, buf.nsel, out, buf.workspace,
                             buf.error_flags)
    torch.cuda.synchronize()
    assert int(buf.error_flags.item()) == 0
    return out


def test_noalloc_decode_equals_the_workspace_decode_on_calls_in_a_row():
    lib = srkv.load()
    large = synth.ragged_batch(n_requests=3, lo=12000, hi=30000, device="cuda", seed=77)
    small = synth.make_case(seq_lens=[9000, 2500], num_q_heads=8, num_kv_heads=2,
                            head_dim=128, init_tokens=512, local_tokens=1024,
                            topk_percent=0.3, dense_boundary=0, seed=79, device="cuda")
    cases = {}
    for name, case in (("large", large), ("small", small)):
        buf = gpu_select(case)
        assert int(buf.error_flags.item()) == 0
        cases[name] = (case, buf, _workspace_out(case, buf))
    for call, name in enumerate(("large", "small", "large", "small")):
        case, buf, want = cases[name]
        out = torch.full_like(want, float("nan"))
        flags = torch.zeros(1, dtype=torch.int32, device="cuda")
        assert _noalloc(lib, case, buf.sel, buf.nsel, out, flags) == 0
        torch.cuda.synchronize()
        assert int(flags.item()) == 0, (call, name)
        assert torch.equal(out, want), (call, name)


def test_noalloc_decode_rejects_a_batch_beyond_its_scratch():
    lib = srkv.load()
    case = synth.llama8b_layer(seq_len=4096, device="cuda", seed=78)
    big = 4096  # requests: far more scratch than the static array holds
    assert srkv.decode_workspace_size(case.cfg, big) > srkv.NOALLOC_WORKSPACE_BYTES
    sel = torch.zeros(big, case.cfg["num_kv_heads"], 1, dtype=torch.int32, device="cuda")
    nsel = torch.zeros(big, case.cfg["num_kv_heads"], dtype=torch.int32, device="cuda")
    table = torch.zeros(big, case.max_blocks, dtype=torch.int32, device="cuda")
    lens = torch.zeros(big, dtype=torch.int32, device="cuda")
    out = torch.zeros(big, case.cfg["num_q_heads"], 128, dtype=torch.bfloat16, device="cuda")
    c = srkv.config(case.cfg)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    status = lib.srkv_sparse_paged_decode_noalloc(
        ctypes.byref(c), p(case.q), p(case.k_cache), p(case.v_cache), case.k_cache.shape[0],
        p(table), case.max_blocks, p(lens), big, p(sel), 1, p(nsel), p(out), None,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert status == 3  # SRKV_ERR_WORKSPACE, returned before any launch
