"""The decode kernels start behind the previous kernel of the stream (programmatic dependent
launch): they must still see every input that kernel wrote.  Here ordinary PyTorch kernels
rewrite the query and the lengths on the same stream right before the call."""
import numpy as np
import pytest
import torch

from block_sparse_retrieval_gb300 import srkv, synth
from parity import check_same, gpu_select

pytestmark = pytest.mark.gpu

DEV = "cuda"


def decode(case, reps, q, seq_lens):
    b = srkv.DecodeBuffers(case.cfg, case.batch, case.max_blocks, case.num_pages, device=DEV)
    b.reps.copy_(reps)
    srkv.retrieval_decode(case.cfg, q, case.k_cache, case.v_cache, b.reps, case.block_table,
                          seq_lens, case.prompt_lens, b.sel, b.nsel, b.out, b.workspace,
                          b.error_flags)
    return b


@pytest.mark.parametrize("name", ["one-kernel", "three-kernel"])
def test_inputs_written_just_before_the_call_are_read(name):
    if name == "one-kernel":
        case = synth.llama8b_layer(seq_len=16384, device=DEV, seed=61)
    else:
        case = synth.ragged_batch(n_requests=5, lo=9000, hi=20000, device=DEV, seed=62)
        assert srkv.retrieval_decode_launches(case.cfg, case.batch, case.max_blocks) == 3
    reps = gpu_select(case).reps
    g = torch.Generator(device=DEV).manual_seed(7)
    q_new = torch.randn(case.q.shape, generator=g, device=DEV).to(case.q.dtype)
    L_new = (case.seq_lens - 300).clamp(min=1)
    want = decode(case, reps, q_new.clone(), L_new.clone())
    torch.cuda.synchronize()
    # the old query and lengths, overwritten by elementwise kernels on the stream
    q = case.q.clone()
    L = case.seq_lens.clone()
    torch.cuda.synchronize()
    for _ in range(3):
        q.mul_(0).add_(q_new)
        L.mul_(0).add_(L_new)
        got = decode(case, reps, q, L)
    torch.cuda.synchronize()
    assert int(got.error_flags.item()) == 0
    assert np.array_equal(got.sel.cpu().numpy(), want.sel.cpu().numpy())
    assert np.array_equal(got.nsel.cpu().numpy(), want.nsel.cpu().numpy())
    check_same(case, got.out.float().cpu().numpy(), want.out.float().cpu().numpy())
    # and not the old query's result
    old = decode(case, reps, case.q, case.seq_lens)
    torch.cuda.synchronize()
    assert not np.allclose(got.out.float().cpu().numpy(), old.out.float().cpu().numpy(), atol=1e-2)
