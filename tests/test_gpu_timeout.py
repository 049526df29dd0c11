"""The bounded-wait abort path on the GPU, made to run without a fault.

A copy of the library is built with a 2 ms wait limit and one wait that
nothing ever completes (MLA_TEST_STALL_WAIT: the score SM's MMA issuer waits
on a barrier that is only arrived on at the end of the kernel).  That wait
gives up, records MLA_STATUS_TIMEOUT and raises the grid-wide abort flag;
every other role leaves its loop; the producers wait until the copies they
issued have landed, the MMA issuers until their MMAs have completed, and the
kernel ends through its normal teardown.  The call must return, the status
must read MLA_STATUS_TIMEOUT (-6), and the normal library must then decode
correctly in the same process (the context is still usable)."""
import os
import tempfile

import numpy as np
import pytest
import torch

from mla_latent_kv_05_gb300 import _build, binding
from mla_latent_kv_05_gb300 import inputs as gen
from oracle import mla_oracle

pytestmark = pytest.mark.gpu

TIMEOUT = -6


@pytest.fixture(scope="module")
def stall_lib():
    d = tempfile.mkdtemp(prefix="mla_stall_")
    path = _build.build(extra_flags=("-DMLA_WAIT_TIMEOUT_NS=2000000ull", "-DMLA_TEST_STALL_WAIT=1"), out_dir=d)
    return binding.load(path)


def _call(lib, name, inp, ws):
    prev = binding._lib
    binding._lib = lib
    try:
        fn = getattr(binding, name)
        return fn(inp.q_absorbed.cuda(), inp.q_rope.cuda(), inp.kv_cache.cuda(), inp.block_table.cuda(),
                  inp.seq_lens.cuda(), inp.scale, workspace=ws)
    finally:
        binding._lib = prev


@pytest.mark.parametrize("kv_dtype,name", [("bf16", "mla_decode_bf16"), ("fp8", "mla_decode_fp8")])
def test_a_wait_that_runs_out_ends_the_call_with_timeout_status(cuda_device, stall_lib, kv_dtype, name):
    inp = gen.make_inputs(2, 1, [300, 300], kv_dtype=kv_dtype, seed=91)
    ws = binding.alloc_workspace(inp.batch, inp.sq)
    _call(stall_lib, name, inp, ws)
    torch.cuda.synchronize()                      # the call returned: no hang
    assert binding.mla_get_status(ws) == TIMEOUT
    # the same context still works: the normal library decodes correctly
    out, lse = _call(binding.load(), name, inp, ws)
    assert binding.mla_get_status(ws) == 0
    rows = mla_oracle.cache_rows(inp.kv_cache.double().numpy() if kv_dtype == "bf16" else inp.kv_cache.numpy(),
                                 kv_dtype)
    ref_out, ref_lse = mla_oracle.mla_decode(inp.q_absorbed.double().numpy(), inp.q_rope.double().numpy(), rows,
                                             inp.block_table.numpy(), inp.seq_lens.numpy(), inp.scale)
    got = out.double().cpu().numpy()
    assert np.abs(got - ref_out).max() <= 1e-2 * np.abs(ref_out).max()
    assert np.abs(lse.double().cpu().numpy() - ref_lse).max() <= 1e-3
