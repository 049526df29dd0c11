"""mla_decode_bf16_noalloc (the decode on the library's own static scratch)
against mla_decode_bf16 with a caller workspace, through the C ABI, and
against the float64 oracle.

Two calls in a row on different problems (a ragged batch whose rows are split
over many CTA pairs, then causal two-token queries), each compared with the
workspace entry point and with the oracle on the same inputs within the
parity tolerance (max|dout| <= 1e-2 * max|ref|, max|dlse| <= 1e-3).  Neither
torch's allocator statistics nor the device's free memory may move across
the calls once the first call has done its set-up (the free-memory reading
is retaken once if another process on the device moved it).  Collected last
so that it also runs after every other GPU test.
"""
import ctypes

import numpy as np
import pytest
import torch

from mla_latent_kv_05_gb300 import binding
from mla_latent_kv_05_gb300 import inputs as gen
from oracle import mla_oracle

pytestmark = pytest.mark.gpu

OUT_RTOL = 1e-2
LSE_ATOL = 1e-3


def _problems():
    a = gen.make_inputs(6, 1, [1, 63, 64, 65, 700, 3000], seed=71)
    b = gen.make_inputs(3, 2, [129, 5000, 2], seed=72, scale=0.07)
    return [a, b]


def _device(inp):
    return (inp.q_absorbed.cuda(), inp.q_rope.cuda(), inp.kv_cache.cuda(), inp.block_table.cuda(),
            inp.seq_lens.cuda())


def _oracle(inp):
    rows = mla_oracle.cache_rows(inp.kv_cache.double().numpy(), "bf16")
    o, l_ = mla_oracle.mla_decode(inp.q_absorbed.double().numpy(), inp.q_rope.double().numpy(), rows,
                                  inp.block_table.numpy(), inp.seq_lens.numpy(), inp.scale)
    return torch.from_numpy(o), torch.from_numpy(l_)


def _compare(out, lse, ref_out, ref_lse):
    got, ref = out.double().cpu().numpy(), ref_out.double().cpu().numpy()
    gl, rl = lse.double().cpu().numpy(), ref_lse.double().cpu().numpy()
    for b in range(got.shape[0]):
        for i in range(got.shape[1]):
            if np.all(np.isneginf(rl[b, i])):
                assert np.all(np.isneginf(gl[b, i])) and np.all(got[b, i] == 0), (b, i)
                continue
            err = np.abs(got[b, i] - ref[b, i]).max()
            assert err <= OUT_RTOL * np.abs(ref[b, i]).max(), (b, i, err)
            assert np.abs(gl[b, i] - rl[b, i]).max() <= LSE_ATOL, (b, i)


def test_noalloc_matches_workspace_entry_on_consecutive_calls(cuda_device):
    probs = _problems()
    dev = [_device(p) for p in probs]
    refs = []
    for p, d in zip(probs, dev):
        ws = binding.alloc_workspace(p.batch, p.sq)
        out, lse = binding.mla_decode_bf16(*d, p.scale, workspace=ws)
        assert binding.mla_get_status(ws) == 0
        refs.append((out, lse))
    outs = [(torch.empty_like(r[0]), torch.empty_like(r[1])) for r in refs]
    status = [torch.full((1,), -99, dtype=torch.int32, device="cuda") for _ in probs]

    # first call on this device: does the one-time set-up
    binding.mla_decode_bf16_noalloc(*dev[0], probs[0].scale, out=outs[0][0], lse=outs[0][1],
                                    device_status=status[0])
    torch.cuda.synchronize()
    assert int(status[0].item()) == 0
    _compare(*outs[0], *refs[0])

    oracles = [_oracle(p) for p in probs]

    def run_both():
        for o in outs:
            o[0].fill_(7)
            o[1].fill_(7)
        for s in status:
            s.fill_(-99)
        torch.cuda.synchronize()
        stats = (torch.cuda.memory_allocated(), torch.cuda.memory_reserved())
        free_before = torch.cuda.mem_get_info()[0]
        for p, d, o, s in zip(probs, dev, outs, status):
            binding.mla_decode_bf16_noalloc(*d, p.scale, out=o[0], lse=o[1], device_status=s)
        torch.cuda.synchronize()
        assert (torch.cuda.memory_allocated(), torch.cuda.memory_reserved()) == stats
        return torch.cuda.mem_get_info()[0] - free_before

    if run_both() != 0:
        # another process may have moved the device's free memory: measure once more
        assert run_both() == 0
    for o, r, orc, s in zip(outs, refs, oracles, status):
        assert int(s.item()) == 0
        _compare(*o, *r)
        _compare(*o, *orc)


def test_noalloc_rejects_rows_beyond_its_scratch(cuda_device):
    lib = binding.load()
    t = torch.zeros(64, dtype=torch.uint8, device="cuda")
    p = ctypes.c_void_p(t.data_ptr())
    # 2049 x 4 = 8196 query rows > 8192: refused on the host before any launch
    rc = lib.mla_decode_bf16_noalloc(p, p, p, p, p, 2049, 4, 128, 8, 64, 4, ctypes.c_float(0.1), p, p, None, None)
    assert rc == -3, binding.status_string(rc)    # MLA_ERR_WORKSPACE
