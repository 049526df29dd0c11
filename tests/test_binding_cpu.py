"""The Python binding's marshalling, run on the CPU against a stand-in for the
library: each wrapper hands the library the pointers, sizes and stream it
should, and refuses tensors on different devices, or on a device other than
the current one, before anything is launched."""
import types

import numpy as np
import pytest
import torch

from mla_latent_kv_05_gb300 import binding


class FakeTensor:
    """Just enough of a CUDA tensor for the wrappers' marshalling."""
    _next = 0x10000

    def __init__(self, shape, dev=0):
        self.shape = tuple(shape)
        self.device = torch.device("cuda", dev)
        FakeTensor._next += 0x10000
        self._ptr = FakeTensor._next

    def dim(self):
        return len(self.shape)

    def numel(self):
        return int(np.prod(self.shape))

    def data_ptr(self):
        return self._ptr


class FakeLib:
    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        def fn(*args):
            self.calls.append((name, args))
            return 0
        return fn


@pytest.fixture
def fake(monkeypatch):
    lib = FakeLib()
    monkeypatch.setattr(binding, "load", lambda *a, **k: lib)
    monkeypatch.setattr(binding, "_check", lambda *a, **k: None)
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    return lib


STREAM = types.SimpleNamespace(cuda_stream=0x77)
B, SQ, H = 3, 2, 128


def _dense(row_bytes, dev_of=None):
    dev_of = dev_of or {}
    t = {
        "q_absorbed": FakeTensor((B, SQ, H, 512), dev_of.get("q_absorbed", 0)),
        "q_rope": FakeTensor((B, SQ, H, 64), dev_of.get("q_rope", 0)),
        "kv_cache": FakeTensor((9, 64, row_bytes), dev_of.get("kv_cache", 0)),
        "block_table": FakeTensor((B, 5), dev_of.get("block_table", 0)),
        "seq_lens": FakeTensor((B,), dev_of.get("seq_lens", 0)),
        "out": FakeTensor((B, SQ, H, 512), dev_of.get("out", 0)),
        "lse": FakeTensor((B, SQ, H), dev_of.get("lse", 0)),
        "workspace": FakeTensor((4096,), dev_of.get("workspace", 0)),
    }
    return t


ENTRIES = [("mla_decode_bf16", 576), ("mla_decode_fp8", 594), ("mla_decode_fp4", 324),
           ("mla_decode_fp8_v41", 528), ("mla_decode_fp4_v41", 288)]


@pytest.mark.parametrize("name,row_bytes", ENTRIES)
def test_dense_wrappers_pass_pointers_sizes_and_stream(fake, name, row_bytes):
    t = _dense(row_bytes)
    out, lse = getattr(binding, name)(t["q_absorbed"], t["q_rope"], t["kv_cache"], t["block_table"], t["seq_lens"],
                                      0.125, out=t["out"], lse=t["lse"], workspace=t["workspace"], stream=STREAM)
    assert out is t["out"] and lse is t["lse"]
    (called, args), = fake.calls
    assert called == name
    ptrs = [a.value for a in args[:5]]
    assert ptrs == [t[k].data_ptr() for k in ("q_absorbed", "q_rope", "kv_cache", "block_table", "seq_lens")]
    assert list(args[5:11]) == [B, SQ, H, 9, 64, 5]           # batch, sq, heads, pages, page size, max_pages
    assert args[11].value == 0.125
    assert [a.value for a in args[12:15]] == [t["out"].data_ptr(), t["lse"].data_ptr(), t["workspace"].data_ptr()]
    assert args[15].value == 4096 and args[16].value == 0x77


@pytest.mark.parametrize("name,row_bytes", ENTRIES)
def test_dense_wrappers_refuse_mixed_or_foreign_devices(fake, name, row_bytes):
    for odd in ("kv_cache", "out", "workspace", "seq_lens"):
        t = _dense(row_bytes, {odd: 1})
        with pytest.raises(ValueError, match=odd):
            getattr(binding, name)(t["q_absorbed"], t["q_rope"], t["kv_cache"], t["block_table"], t["seq_lens"],
                                   0.125, out=t["out"], lse=t["lse"], workspace=t["workspace"], stream=STREAM)
    t = _dense(row_bytes, {k: 1 for k in ("q_absorbed", "q_rope", "kv_cache", "block_table", "seq_lens", "out",
                                          "lse", "workspace")})
    with pytest.raises(ValueError, match="current device"):
        getattr(binding, name)(t["q_absorbed"], t["q_rope"], t["kv_cache"], t["block_table"], t["seq_lens"],
                               0.125, out=t["out"], lse=t["lse"], workspace=t["workspace"], stream=STREAM)
    assert fake.calls == []


def test_noalloc_sparse_wuv_and_merge_wrappers(fake):
    t = _dense(576)
    status = FakeTensor((1,))
    binding.mla_decode_bf16_noalloc(t["q_absorbed"], t["q_rope"], t["kv_cache"], t["block_table"], t["seq_lens"],
                                    0.1, out=t["out"], lse=t["lse"], device_status=status, stream=STREAM)
    slots = FakeTensor((B, SQ, 100))
    binding.mla_decode_sparse_bf16(t["q_absorbed"], t["q_rope"], t["kv_cache"], slots, 0.1, out=t["out"],
                                   lse=t["lse"], workspace=t["workspace"], stream=STREAM)
    lat, w, up = FakeTensor((B, SQ, 128, 512)), FakeTensor((128, 128, 512)), FakeTensor((B, SQ, 128, 128))
    binding.mla_up_project_wuv(lat, w, out=up, workspace=FakeTensor((256,)), stream=STREAM)
    po, pl, ip = FakeTensor((7, 128, 512)), FakeTensor((7, 128)), FakeTensor((5,))
    binding.mla_combine_splits(po, pl, ip, out=FakeTensor((4, 128, 512)), lse=FakeTensor((4, 128)), stream=STREAM)
    names = [c[0] for c in fake.calls]
    assert names == ["mla_decode_bf16_noalloc", "mla_decode_sparse_bf16", "mla_up_project_wuv", "mla_combine_splits"]
    noalloc, sparse, wuv, comb = [c[1] for c in fake.calls]
    assert noalloc[14].value == status.data_ptr() and noalloc[15].value == 0x77
    assert list(sparse[4:10]) == [B, SQ, 100, H, 9, 64]        # batch, sq, topk, heads, pages, page size
    assert wuv[2:5] == (B * SQ, 128, 128)
    assert comb[3:5] == (4, 128)                               # rows, heads

    with pytest.raises(ValueError, match="token_slots"):
        binding.mla_decode_sparse_bf16(t["q_absorbed"], t["q_rope"], t["kv_cache"], FakeTensor((B, SQ, 100), 1),
                                       0.1, out=t["out"], lse=t["lse"], workspace=t["workspace"], stream=STREAM)
    with pytest.raises(ValueError, match="w_uv"):
        binding.mla_up_project_wuv(lat, FakeTensor((128, 128, 512), 1), out=up, workspace=FakeTensor((256,)),
                                   stream=STREAM)
    with pytest.raises(ValueError, match="partial_out"):
        binding.mla_combine_splits(FakeTensor((7, 128, 64)), pl, ip, out=FakeTensor((4, 128, 512)),
                                   lse=FakeTensor((4, 128)), stream=STREAM)
    with pytest.raises(ValueError, match="split_indptr"):
        binding.mla_combine_splits(po, pl, FakeTensor((5, 1)), stream=STREAM)
    assert len(fake.calls) == 4
