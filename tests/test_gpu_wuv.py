"""GPU parity of the W^UV up-projection (through the C ABI) against the
float64 oracle, alone (ragged row counts across 128-row tiles) and after the
decode: absorbed decode + up-projection on the GPU against the oracle's
un-absorbed attention with explicit per-head W^UK and W^UV (the guide's
matrix-absorption identity, end to end).

Bound: max|out - ref| <= 1e-2 * max|ref| per head row block.
"""
import numpy as np
import pytest
import torch

from mla_latent_kv_05_gb300 import binding
from mla_latent_kv_05_gb300 import inputs as gen
from oracle import mla_oracle

pytestmark = pytest.mark.gpu


def _w(gen_, shape, scale):
    return (torch.randn(shape, generator=gen_) * scale).to(torch.bfloat16)


@pytest.mark.parametrize("rows", [1, 64, 130, 300])
def test_up_projection_matches_oracle(cuda_device, rows):
    g = torch.Generator().manual_seed(70 + rows)
    latent = _w(g, (rows, 128, 512), 1.0)
    w_uv = _w(g, (128, 128, 512), 512 ** -0.5)
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    out = binding.mla_up_project_wuv(latent.cuda(), w_uv.cuda(), workspace=ws)
    assert binding.mla_get_status(ws) == 0
    ref = np.stack([mla_oracle.up_project_output(latent[r].double().numpy(), w_uv.double().numpy())
                    for r in range(rows)])
    got = out.double().cpu().numpy()
    err = np.abs(got - ref).max()
    assert err <= 1e-2 * np.abs(ref).max(), err


def test_absorbed_decode_then_up_projection_equals_unabsorbed_attention(cuda_device):
    # per head: k_j = W^UK c_j, v_j = W^UV c_j, q_abs = (W^UK)^T q
    g = torch.Generator().manual_seed(77)
    d = gen.make_inputs(2, 1, [150, 70], seed=78)
    w_uk = _w(g, (128, 128, 512), 512 ** -0.5)
    w_uv = _w(g, (128, 128, 512), 512 ** -0.5)
    q_nope = _w(g, (2, 1, 128, 128), 1.0)
    q_abs = torch.from_numpy(np.stack([[mla_oracle.absorb_query(q_nope[b, 0].double().numpy(),
                                                                w_uk.double().numpy())] for b in range(2)]))
    d.q_absorbed = q_abs.to(torch.bfloat16)
    out_lat, _ = binding.mla_decode_bf16(d.q_absorbed.cuda(), d.q_rope.cuda(), d.kv_cache.cuda(),
                                         d.block_table.cuda(), d.seq_lens.cuda(), d.scale)
    out = binding.mla_up_project_wuv(out_lat, w_uv.cuda()).double().cpu().numpy()
    rows = mla_oracle.cache_rows(d.kv_cache.double().numpy(), "bf16")
    for b in range(2):
        n = int(d.seq_lens[b])
        c = mla_oracle.gather_rows(rows, d.block_table[b].numpy(), n)
        # the un-absorbed reference uses the bf16-rounded absorbed query's own
        # source (q_nope) and weights: the absorption identity is exact in
        # real arithmetic, so the only differences are the GPU's roundings
        ref, _ = mla_oracle.attend_unabsorbed(q_nope[b, 0].double().numpy(), d.q_rope[b, 0].double().numpy(),
                                              c[:, :512], c[:, 512:], w_uk.double().numpy(),
                                              w_uv.double().numpy(), d.scale)
        # the same bound as everywhere else: the GPU's roundings (the bf16
        # absorbed query, the bf16 latent output, the bf16 result) give about
        # 3e-3 to 5e-3 of max|ref| on these inputs
        err = np.abs(out[b, 0] - ref).max()
        assert err <= 1e-2 * np.abs(ref).max(), (b, err)
