"""The C-ABI library builds, loads, and exports every symbol include/dsa.h
declares; host-side validation rejects bad arguments before touching a GPU.
No compute call is made here (no GPU needed)."""
import ctypes
import os
import re
import subprocess

import pytest

from kv_cache_serving_gb300 import build, dsa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsa.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_[a-z_]+)\s*\(", text)))


def test_header_declares_the_path():
    names = declared_functions()
    for want in ("dsa_build_index", "dsa_decode_sparse", "dsa_decode_sparse_masked",
                 "dsa_decode_dense",
                 "dsa_attention_mass", "dsa_workspace_size", "dsa_status_string",
                 "dsa_get_device_error"):
        assert want in names


def test_library_exports_every_declared_symbol():
    lib = build.build()
    out = subprocess.run(["nm", "-D", "--defined-only", lib], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\s[TW]\s+(dsa_\w+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    # C linkage: no mangled dsa entry points leak out as the only definition
    assert all(not n.startswith("_Z") for n in exported)


def test_tuning_setters():
    for setter, getter, good, bad in (
            (dsa.dsa_set_sparse_cluster, dsa.dsa_get_sparse_cluster, (0, 1, 2, 8), (-1, 9)),
            (dsa.dsa_set_prefill_split, dsa.dsa_get_prefill_split, (0, 1, 2, 8), (-1, 9)),):
        saved = getter()
        try:
            for v in good:
                setter(v)
                assert getter() == v
            for v in bad:
                with pytest.raises(dsa.DSAError):
                    setter(v)
        finally:
            setter(saved)


def test_host_only_calls():
    assert dsa.dsa_version() >= 1
    assert dsa.dsa_status_string(0) == "DSA_OK"
    assert dsa.dsa_status_string(4) == "DSA_ERR_DEVICE"
    assert dsa.dsa_status_string(99) == "DSA_ERR_UNKNOWN"
    d = dsa.make_dims(4, 8, 2, 128, 100, 20, 96, 3, 400, "bf16", "bf16")
    n = dsa.dsa_workspace_size(d)
    assert n >= 256 + 4 * 8 * (128 + 2) * 4
    assert n % 4 == 0


@pytest.mark.parametrize("field,value,status", [
    ("head_dim", 96, dsa.DSA_ERR_UNSUPPORTED),
    ("page_size", 32, dsa.DSA_ERR_UNSUPPORTED),
    ("hq", 6, dsa.DSA_ERR_INVALID_ARG),        # not a multiple of hkv=4
    ("hq", 48, dsa.DSA_ERR_UNSUPPORTED),       # group 12 not built
    ("mask_words", 2, dsa.DSA_ERR_INVALID_ARG),  # 64 bits < max_window 96
    ("max_kept", 0, dsa.DSA_ERR_INVALID_ARG),
    ("kv_dtype", 7, dsa.DSA_ERR_INVALID_ARG),
])
def test_dims_validation(field, value, status):
    d = dsa.make_dims(2, 8, 4, 128, 10, 4, 96, 3, 50, "bf16", "bf16")
    setattr(d, field, value)
    lib = dsa._load()
    assert lib.dsa_workspace_size(ctypes.byref(d)) == 0
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: validation fails first
    st = lib.dsa_decode_dense(ctypes.byref(d), fake, fake, fake, fake, fake, 0.1, fake, None,
                              fake, None)
    assert st == status


def test_null_pointers_rejected_before_launch():
    lib = dsa._load()
    d = dsa.make_dims(2, 8, 4, 128, 10, 4, 96, 3, 50, "bf16", "bf16")
    fake = ctypes.c_void_p(1 << 20)
    D = ctypes.byref(d)
    assert lib.dsa_decode_sparse(D, fake, fake, fake, fake, fake, None, fake, 0.1, fake, None,
                                 fake, None) == dsa.DSA_ERR_INVALID_ARG
    assert lib.dsa_build_index(D, fake, fake, None, fake, fake, fake, fake, None) == \
        dsa.DSA_ERR_INVALID_ARG
    assert lib.dsa_attention_mass(D, fake, fake, fake, fake, fake, fake, fake, -1, 2, 0.1, fake,
                                  None, fake, None) == dsa.DSA_ERR_INVALID_ARG
    # misaligned workspace
    assert lib.dsa_decode_dense(D, fake, fake, fake, fake, fake, 0.1, fake, None,
                                ctypes.c_void_p((1 << 20) + 8), None) == dsa.DSA_ERR_INVALID_ARG
    # masked decode: a missing keep mask, then a window too long for the in-kernel list
    assert lib.dsa_decode_sparse_masked(D, fake, fake, fake, fake, fake, fake, fake, None, None,
                                        None, None, 0.1, fake, None, fake,
                                        None) == dsa.DSA_ERR_INVALID_ARG
    # an appended K row without its V row
    assert lib.dsa_decode_sparse_masked(D, fake, fake, fake, fake, fake, fake, fake, fake, None,
                                        fake, None, 0.1, fake, None, fake,
                                        None) == dsa.DSA_ERR_INVALID_ARG
    big = dsa.make_dims(2, 8, 4, 128, 10, 4, 1025, 33, 50, "bf16", "bf16")
    assert lib.dsa_decode_sparse_masked(ctypes.byref(big), fake, fake, fake, fake, fake, fake,
                                        fake, fake, None, None, None, 0.1, fake, None, fake,
                                        None) == \
        dsa.DSA_ERR_UNSUPPORTED
    assert lib.dsa_decode_plan(ctypes.byref(d), 3, None, None, None, None, None) == \
        dsa.DSA_ERR_INVALID_ARG
    # eviction: a missing free-list counter, a negative capacity
    assert lib.dsa_evict_pages(D, fake, fake, fake, fake, fake, None, 4, fake,
                               None) == dsa.DSA_ERR_INVALID_ARG
    assert lib.dsa_evict_pages(D, fake, fake, fake, fake, fake, fake, -1, fake,
                               None) == dsa.DSA_ERR_INVALID_ARG
    code = ctypes.c_int32(0)
    assert lib.dsa_get_device_error(None, None, ctypes.byref(code)) == dsa.DSA_ERR_INVALID_ARG


def test_prefill_call_checks_before_launch():
    """dsa_prefill_sparse: host checks (no GPU): a missing q_len, a negative
    max_q, fp32 KV or a window past 32768 are refused; max_q = 0 or an empty
    batch is a no-op that touches nothing."""
    lib = dsa._load()
    fake = ctypes.c_void_p(1 << 20)
    d = dsa.make_dims(2, 8, 2, 128, 10, 4, 96, 3, 50, "bf16", "bf16")
    D = ctypes.byref(d)

    def call(dims=D, max_q=4, q_len=fake):
        return lib.dsa_prefill_sparse(dims, max_q, fake, fake, fake, fake, fake, q_len, fake,
                                      fake, fake, None, 0.1, fake, None, fake, None)
    assert call(q_len=None) == dsa.DSA_ERR_INVALID_ARG
    assert call(max_q=-1) == dsa.DSA_ERR_INVALID_ARG
    assert call(max_q=0) == dsa.DSA_OK
    f32 = dsa.make_dims(2, 8, 2, 128, 10, 4, 96, 3, 50, "bf16", "f32")
    assert call(dims=ctypes.byref(f32)) == dsa.DSA_ERR_UNSUPPORTED
    wide = dsa.make_dims(2, 8, 2, 128, 10, 4, 32769, 1025, 50, "bf16", "bf16")
    assert call(dims=ctypes.byref(wide)) == dsa.DSA_ERR_UNSUPPORTED
    empty = dsa.make_dims(0, 8, 2, 128, 10, 4, 96, 3, 50, "bf16", "bf16")
    assert call(dims=ctypes.byref(empty)) == dsa.DSA_OK
    # the plan query makes the same argument checks before it asks the device
    assert lib.dsa_prefill_plan(D, -1, None, None, None, None, None, None) == dsa.DSA_ERR_INVALID_ARG
    assert (lib.dsa_prefill_plan(ctypes.byref(f32), 4, None, None, None, None, None, None)
            == dsa.DSA_ERR_UNSUPPORTED)
    w = ctypes.c_int32(-1)
    assert lib.dsa_prefill_plan(D, 0, ctypes.byref(w), None, None, None, None, None) == dsa.DSA_OK
    assert w.value == 2


def test_host_io_call_checks_before_copying():
    """dsa_decode_sparse_masked_io rejects a bad call before its upload: no io,
    an io copy without its buffers, or bad decode arguments (the fake pointers
    are never dereferenced, so nothing reaches a GPU)."""
    lib = dsa._load()
    d = dsa.make_dims(2, 8, 4, 128, 10, 4, 96, 3, 50, "bf16", "bf16")
    fake = ctypes.c_void_p(1 << 20)
    D = ctypes.byref(d)
    ok_io = dsa.dsa_host_io(1 << 20, 1 << 21, 256, 1 << 22, 1 << 23, 256)

    def call(io, keep_mask=fake, dims=D):
        return lib.dsa_decode_sparse_masked_io(io, dims, fake, fake, fake, fake, fake, fake, fake,
                                               keep_mask, None, None, None, 0.1, fake, None,
                                               fake, None)
    assert call(None) == dsa.DSA_ERR_INVALID_ARG
    for field in ("host_in", "dev_in", "dev_out", "host_out"):
        io = dsa.dsa_host_io(1 << 20, 1 << 21, 256, 1 << 22, 1 << 23, 256)
        setattr(io, field, None)
        assert call(ctypes.byref(io)) == dsa.DSA_ERR_INVALID_ARG, field
    # bad decode arguments with a valid io: rejected before the upload
    assert call(ctypes.byref(ok_io), keep_mask=None) == dsa.DSA_ERR_INVALID_ARG
    big = dsa.make_dims(2, 8, 4, 128, 10, 4, 1025, 33, 50, "bf16", "bf16")
    assert call(ctypes.byref(ok_io), dims=ctypes.byref(big)) == dsa.DSA_ERR_UNSUPPORTED


def test_graph_handles_checked():
    lib = dsa._load()
    assert lib.dsa_graph_launch(None, None) == dsa.DSA_ERR_INVALID_ARG
    assert lib.dsa_graph_destroy(None) == dsa.DSA_OK
    assert lib.dsa_graph_begin(None) == dsa.DSA_ERR_INVALID_ARG   # legacy stream
    assert lib.dsa_graph_end(None, None) == dsa.DSA_ERR_INVALID_ARG


def test_prepared_call_reissues_and_raises():
    """dsa.Prepared keeps the marshalled arguments and re-issues the call;
    a non-OK status raises (host-only entry point, no GPU)."""
    saved = dsa.dsa_get_sparse_cluster()
    try:
        set4 = dsa.Prepared("dsa_set_sparse_cluster", (ctypes.c_int32(4),))
        dsa.dsa_set_sparse_cluster(0)
        set4()
        assert dsa.dsa_get_sparse_cluster() == 4
        dsa.dsa_set_sparse_cluster(1)
        set4()
        assert dsa.dsa_get_sparse_cluster() == 4
        with pytest.raises(dsa.DSAError):
            dsa.Prepared("dsa_set_sparse_cluster", (ctypes.c_int32(-1),))()
    finally:
        dsa.dsa_set_sparse_cluster(saved)


def test_host_io_binding_checks_buffers():
    import torch
    a = torch.zeros(64, dtype=torch.uint8)
    with pytest.raises(TypeError):
        dsa.host_io(a, a, a, a)   # device sides must be CUDA tensors
    with pytest.raises(TypeError):
        dsa.dsa_decode_sparse_masked_io(None, None, *([None] * 10))
