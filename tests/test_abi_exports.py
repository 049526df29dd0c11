"""The C-ABI library builds, loads without a GPU, exports every entry point
include/mla_decode.h declares, and rejects bad arguments on the host before
touching CUDA."""
import ctypes
import os
import re

import pytest

from mla_latent_kv_05_gb300 import _build, binding

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "mla_decode.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return binding.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_expected_entry_points():
    names = declared_functions()
    for n in ("mla_decode_bf16", "mla_decode_fp8", "mla_decode_fp4", "mla_combine_splits", "mla_workspace_size",
              "mla_get_status", "mla_status_string", "mla_decode_sparse_bf16", "mla_workspace_size_sparse"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) <= set(binding.SIGNATURES)


def _declarations():
    """name -> (return type, [argument types]) from the header's prototypes."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {}
    for m in re.finditer(r"([A-Za-z_][A-Za-z0-9_ *]*?)\b(mla_[a-z0-9_]+)\s*\(([^)]*)\)\s*;", text):
        args = [" ".join(a.split()) for a in m.group(3).split(",")] if m.group(3).strip() else []
        # drop each argument's name, keep its type (with any '*')
        types = [re.sub(r"\s*\b[A-Za-z_][A-Za-z0-9_]*$", "", a).replace(" *", "*") for a in args]
        out[m.group(2)] = (" ".join(m.group(1).split()).replace(" *", "*"), types)
    return out


def _ctype_of(c_type):
    c_type = c_type.replace("const ", "")
    if c_type == "int":
        return ctypes.c_int
    if c_type == "float":
        return ctypes.c_float
    if c_type == "size_t":
        return ctypes.c_size_t
    if c_type == "size_t*":
        return ctypes.POINTER(ctypes.c_size_t)
    if c_type == "char*":
        return ctypes.c_char_p
    if c_type.endswith("*"):
        return ctypes.c_void_p
    raise AssertionError("unmapped C type " + c_type)


def test_binding_signatures_match_the_header_argument_by_argument():
    decls = _declarations()
    assert set(decls) == set(binding.SIGNATURES)
    for name, (ret, args) in decls.items():
        res, argtypes = binding.SIGNATURES[name]
        assert res is _ctype_of(ret), name
        assert len(argtypes) == len(args), name
        for i, (want, got) in enumerate(zip(args, argtypes)):
            w = _ctype_of(want)
            same = got is w or (hasattr(w, "_type_") and getattr(got, "_type_", None) is w._type_)
            assert same, (name, i, want, got)


def test_status_codes_match_the_header():
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    codes = {int(v): k for k, v in re.findall(r"\b(MLA_[A-Z_]+)\s*=\s*(-?\d+)", text)}
    assert codes == binding._STATUS


def test_status_strings(lib):
    for code, name in binding._STATUS.items():
        assert lib.mla_status_string(code).decode() == name


def test_host_validation_without_gpu(lib):
    z = ctypes.c_void_p(0)
    rc = lib.mla_decode_bf16(z, z, z, z, z, 1, 1, 128, 8, 64, 4, ctypes.c_float(0.1), z, z, z, 0, z)
    assert rc == -1
    n = ctypes.c_size_t(0)
    assert lib.mla_workspace_size(1, 1, 64, 64, ctypes.byref(n)) == -2     # num_heads != 128
    assert lib.mla_workspace_size(1, 1, 128, 32, ctypes.byref(n)) == -2    # page_size != 64
    assert lib.mla_workspace_size(1, 5, 128, 64, ctypes.byref(n)) == -2    # Sq > 4
    assert lib.mla_workspace_size(1, 0, 128, 64, ctypes.byref(n)) == -1
    assert lib.mla_combine_splits(z, z, z, -1, 128, z, z, z) == -1
    fake = ctypes.c_void_p(0x1000)
    rc = lib.mla_decode_bf16(fake, fake, fake, fake, fake, 1, 1, 64, 8, 64, 4, ctypes.c_float(0.1),
                             fake, fake, fake, 1 << 30, z)
    assert rc == -2
    rc = lib.mla_decode_fp8(fake, fake, fake, fake, fake, 1, 1, 128, 8, 64, 4, ctypes.c_float(float("nan")),
                            fake, fake, fake, 1 << 30, z)
    assert rc == -1
    rc = lib.mla_decode_fp4(fake, fake, fake, fake, fake, 1, 1, 128, 8, 64, 4, ctypes.c_float(float("inf")),
                            fake, fake, fake, 1 << 30, z)
    assert rc == -1
    rc = lib.mla_decode_fp4(fake, fake, ctypes.c_void_p(0x1004), fake, fake, 1, 1, 128, 8, 64, 4,
                            ctypes.c_float(0.1), fake, fake, fake, 1 << 30, z)   # cache not 16-byte aligned
    assert rc == -1
    for bad_scale in (0.0, -0.1):
        rc = lib.mla_decode_bf16(fake, fake, fake, fake, fake, 1, 1, 128, 8, 64, 4, ctypes.c_float(bad_scale),
                                 fake, fake, fake, 1 << 30, z)
        assert rc == -1


def test_sparse_host_validation_without_gpu(lib):
    z = ctypes.c_void_p(0)
    fake = ctypes.c_void_p(0x1000)
    n = ctypes.c_size_t(0)
    assert lib.mla_workspace_size_sparse(1, 1, 0, 128, 64, ctypes.byref(n)) == -1        # topk = 0
    assert lib.mla_workspace_size_sparse(1, 1, 1 << 15, 128, 64, ctypes.byref(n)) == -2  # topk > 16384
    assert lib.mla_workspace_size_sparse(1, 1, 64, 64, 64, ctypes.byref(n)) == -2        # num_heads != 128
    rc = lib.mla_decode_sparse_bf16(z, z, z, z, 1, 1, 64, 128, 8, 64, ctypes.c_float(0.1), z, z, z, 0, z)
    assert rc == -1
    rc = lib.mla_decode_sparse_bf16(fake, fake, fake, fake, 1, 1, 64, 128, 8, 32, ctypes.c_float(0.1),
                                    fake, fake, fake, 1 << 30, z)
    assert rc == -2                                                                   # page_size != 64
    rc = lib.mla_decode_sparse_bf16(fake, fake, fake, fake, 1, 1, 64, 128, 8, 64, ctypes.c_float(float("inf")),
                                    fake, fake, fake, 1 << 30, z)
    assert rc == -1


DENSE_ENTRIES = ["mla_decode_bf16", "mla_decode_fp8", "mla_decode_fp4", "mla_decode_fp8_v41", "mla_decode_fp4_v41"]


@pytest.mark.parametrize("name", DENSE_ENTRIES)
def test_every_dense_entry_validates_on_the_host(lib, name):
    """Each dense decode entry checks its arguments before touching CUDA:
    the same codes from every cache format."""
    fn = getattr(lib, name)
    z = ctypes.c_void_p(0)
    fake = ctypes.c_void_p(0x1000)

    def call(q=fake, cache=fake, batch=1, sq=1, heads=128, pages=8, page=64, max_pages=4, scale=0.1, ws=fake):
        return fn(q, fake, cache, fake, fake, batch, sq, heads, pages, page, max_pages, ctypes.c_float(scale),
                  fake, fake, ws, 1 << 30, z)

    assert call(q=z) == -1                                   # null pointer
    assert call(ws=z) == -1
    assert call(batch=-1) == -1
    assert call(sq=0) == -1
    assert call(max_pages=0) == -1
    assert call(scale=float("nan")) == -1
    assert call(scale=0.0) == -1
    assert call(cache=ctypes.c_void_p(0x1008)) == -1         # cache not 16-byte aligned
    assert call(ws=ctypes.c_void_p(0x1080)) == -1            # workspace not 256-byte aligned
    assert call(heads=64) == -2
    assert call(page=32) == -2
    assert call(sq=5) == -2
    assert call(batch=1 << 15, sq=4) == -2                   # more query rows than the planner takes
    assert call(batch=0) == 0                                # nothing to do: returns before any launch


def test_up_projection_merge_and_profiling_entries_validate_on_the_host(lib):
    z = ctypes.c_void_p(0)
    fake = ctypes.c_void_p(0x1000)
    wuv = lib.mla_up_project_wuv
    assert wuv(z, fake, 4, 128, 128, fake, fake, 1 << 20, z) == -1          # null latent
    assert wuv(fake, fake, -1, 128, 128, fake, fake, 1 << 20, z) == -1      # negative rows
    assert wuv(fake, fake, 4, 64, 128, fake, fake, 1 << 20, z) == -2        # num_heads != 128
    assert wuv(fake, fake, 4, 128, 64, fake, fake, 1 << 20, z) == -2        # d_v != 128
    assert wuv(fake, fake, (1 << 16) + 1, 128, 128, fake, fake, 1 << 20, z) == -2
    assert wuv(fake, ctypes.c_void_p(0x1002), 4, 128, 128, fake, fake, 1 << 20, z) == -1   # W^UV not 16-byte aligned
    assert wuv(fake, fake, 4, 128, 128, fake, fake, 8, z) == -3             # workspace smaller than its header
    assert wuv(fake, fake, 0, 128, 128, fake, fake, 1 << 20, z) == 0        # no rows: nothing launched
    comb = lib.mla_combine_splits
    assert comb(fake, fake, fake, 3, 64, fake, fake, z) == -2               # num_heads != 128
    assert comb(z, fake, fake, 3, 128, fake, fake, z) == -1                 # null partials
    assert comb(ctypes.c_void_p(0x1004), fake, fake, 3, 128, fake, fake, z) == -1
    assert comb(z, z, fake, 0, 128, fake, fake, z) == 0                     # no rows
    assert lib.mla_profile_next_decode(fake, z) == -1                       # both events or neither
    assert lib.mla_profile_next_decode(z, z) == 0
    assert lib.mla_get_status(z, z) == -1
