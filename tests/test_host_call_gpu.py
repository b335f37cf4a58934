"""srkv_retrieval_decode_host: the query and lengths from host memory, the output into host
memory, against srkv_retrieval_decode on the same inputs: the same selection, and the same
output (to the bit where every kept block goes out with the release, so the partial sums
split at fixed pages; within the path-against-path tolerance where the streaming CTAs take
kept blocks from the shared pool)."""
import numpy as np
import pytest
import torch

from block_sparse_retrieval_gb300 import srkv, synth
from parity import check_same, gpu_select

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _device_call(case, buf):
    srkv.retrieval_decode(case.cfg, case.q, case.k_cache, case.v_cache, buf.reps,
                          case.block_table, case.seq_lens, case.prompt_lens, buf.sel, buf.nsel,
                          buf.out, buf.workspace, buf.error_flags)
    torch.cuda.synchronize()
    return buf.out.cpu().clone(), buf.sel.cpu().clone(), buf.nsel.cpu().clone()


@pytest.mark.parametrize("name,pinned,bitwise", [("llama8b-16k", True, True),
                                                 ("ragged-4", True, False),
                                                 ("ragged-4", False, False)])
def test_host_call_matches_the_device_call(name, pinned, bitwise):
    # llama8b-16k: 8 units on clusters of 12, 64 kept blocks each (<= 16 per streaming CTA);
    # ragged-4: 32 units on clusters of 4, prompts below DENSE_BOUNDARY keep all 18-59
    # candidates (up to more than 16 per streaming CTA)
    case = {"llama8b-16k": lambda: synth.llama8b_layer(seq_len=16384, device=DEV),
            "ragged-4": lambda: synth.ragged_batch(n_requests=4, lo=9000, hi=20000,
                                                   device=DEV)}[name]()
    buf = gpu_select(case)
    want_out, want_sel, want_nsel = _device_call(case, buf)
    assert int(buf.error_flags.item()) == 0

    def host(t):
        t = t.cpu().contiguous()
        return t.pin_memory() if pinned else t
    q_host, lens_host = host(case.q), host(case.seq_lens)
    prompt_host = host(case.prompt_lens) if case.prompt_lens is not None else None
    out_host = host(torch.zeros_like(buf.out))
    staging = torch.full((srkv.host_staging_size(case.cfg, case.batch),), 0xFF,
                         dtype=torch.uint8, device=DEV)
    buf.out.fill_(float("nan"))
    buf.sel.fill_(-7)
    srkv.retrieval_decode_host(case.cfg, q_host, lens_host, prompt_host, out_host, staging,
                               case.k_cache, case.v_cache, buf.reps, case.block_table, buf.sel,
                               buf.nsel, buf.out, buf.workspace, buf.error_flags)
    # returns with the output in host memory: no synchronisation needed before reading it
    assert int(buf.error_flags.item()) == 0
    if bitwise:
        assert torch.equal(out_host.view(torch.int16), want_out.view(torch.int16))
    else:
        check_same(case, out_host.float().numpy(), want_out.float().numpy())
    for r in range(case.batch):
        for h in range(case.cfg["num_kv_heads"]):
            k = int(want_nsel[r, h])
            assert int(buf.nsel[r, h]) == k
            assert np.array_equal(buf.sel[r, h, :k].cpu().numpy(), want_sel[r, h, :k].numpy())


def test_host_call_with_inputs_in_one_buffer():
    """Inputs laid out like the staging (srkv.host_inputs) go in one copy: same output."""
    case = synth.ragged_batch(n_requests=3, lo=9000, hi=20000, seed=21, device=DEV)
    buf = gpu_select(case)
    want_out, _, want_nsel = _device_call(case, buf)
    hin = srkv.host_inputs(case.cfg, case.batch)
    hin["q"].copy_(case.q.cpu())
    hin["seq_lens"].copy_(case.seq_lens.cpu())
    hin["prompt_lens"].copy_(case.prompt_lens.cpu())
    out_host = torch.zeros(buf.out.shape, dtype=buf.out.dtype).pin_memory()
    staging = torch.full((srkv.host_staging_size(case.cfg, case.batch),), 0xFF,
                         dtype=torch.uint8, device=DEV)
    buf.nsel.fill_(-1)
    srkv.retrieval_decode_host(case.cfg, hin["q"], hin["seq_lens"], hin["prompt_lens"],
                               out_host, staging, case.k_cache, case.v_cache, buf.reps,
                               case.block_table, buf.sel, buf.nsel, buf.out, buf.workspace,
                               buf.error_flags)
    assert int(buf.error_flags.item()) == 0
    assert torch.equal(buf.nsel.cpu(), want_nsel)
    check_same(case, out_host.float().numpy(), want_out.float().numpy())
    # the staging now holds the query and lengths as the inputs had them
    got = staging.cpu()
    qb = case.q.numel() * 2
    assert torch.equal(got[:qb], hin["q"].view(-1).view(torch.uint8))
    lo = (qb + 255) // 256 * 256
    assert torch.equal(got[lo:lo + 4 * case.batch].view(torch.int32), case.seq_lens.cpu())


def test_marshal_once_step_matches_the_call():
    """srkv.HostDecodeStep (arguments checked and marshalled once) runs the same call: new
    inputs written into the same host buffers give the new step's output."""
    case = synth.llama8b_layer(seq_len=16384, device=DEV)
    buf = gpu_select(case)
    hin = srkv.host_inputs(case.cfg, case.batch)
    out_host = torch.zeros(buf.out.shape, dtype=buf.out.dtype).pin_memory()
    staging = torch.empty(srkv.host_staging_size(case.cfg, case.batch), dtype=torch.uint8,
                          device=DEV)
    step = srkv.HostDecodeStep(case.cfg, hin["q"], hin["seq_lens"], hin["prompt_lens"],
                               out_host, staging, case.k_cache, case.v_cache, buf.reps,
                               case.block_table, buf.sel, buf.nsel, buf.out, buf.workspace,
                               buf.error_flags)
    for scale in (1.0, -0.5):  # two steps: the second with another query, same buffers
        q = (case.q.float() * scale).to(case.q.dtype)
        hin["q"].copy_(q.cpu())
        hin["seq_lens"].copy_(case.seq_lens.cpu())
        hin["prompt_lens"].copy_(case.prompt_lens.cpu())
        step()
        got = out_host.clone()
        ref = srkv.DecodeBuffers(case.cfg, case.batch, case.max_blocks, case.num_pages,
                                 device=DEV)
        ref.reps.copy_(buf.reps)
        srkv.retrieval_decode(case.cfg, q, case.k_cache, case.v_cache, ref.reps,
                              case.block_table, case.seq_lens, case.prompt_lens, ref.sel,
                              ref.nsel, ref.out, ref.workspace, ref.error_flags)
        torch.cuda.synchronize()
        assert int(buf.error_flags.item()) == 0 and int(ref.error_flags.item()) == 0
        # 8 units on clusters of 12, every kept block with the release: the same bits
        assert torch.equal(got.view(torch.int16), ref.out.cpu().view(torch.int16))


def test_host_call_rejects_a_device_query():
    case = synth.llama8b_layer(seq_len=16384, device=DEV)
    buf = gpu_select(case)
    staging = torch.empty(srkv.host_staging_size(case.cfg, case.batch), dtype=torch.uint8,
                          device=DEV)
    with pytest.raises(ValueError):
        srkv.retrieval_decode_host(case.cfg, case.q, case.seq_lens.cpu(), None,
                                   torch.empty(buf.out.shape, dtype=buf.out.dtype), staging,
                                   case.k_cache, case.v_cache, buf.reps, case.block_table,
                                   buf.sel, buf.nsel, buf.out, buf.workspace)
