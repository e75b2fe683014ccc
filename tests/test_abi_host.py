"""The C-ABI library builds, loads and exports every symbol include/mla_nvfp4.h
declares; host-side validation rejects bad arguments before any launch.

CPU only: no call here reaches a CUDA launch (every call below fails
validation, or is a pure host query)."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mla_nvfp4.h")


@pytest.fixture(scope="module")
def lib():
    from sparse_mla_decode_kv_gb300 import build
    build.build()
    import sparse_mla_decode_kv_gb300 as m
    return m.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported_and_bound(lib):
    import sparse_mla_decode_kv_gb300 as m
    names = declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), f"{n} declared but not exported"
        assert n in m.SIGNATURES, f"{n} has no Python binding"
    assert set(m.SIGNATURES) == set(names)


def test_row_bytes_and_status_strings(lib):
    assert lib.mla_kv_row_bytes(0) == 352
    assert lib.mla_kv_row_bytes(1) == 576
    assert lib.mla_kv_row_bytes(7) == 0
    assert lib.mla_status_string(0) == b"MLA_OK"
    assert lib.mla_status_string(3) == b"MLA_ERR_WORKSPACE_TOO_SMALL"
    err = C.c_int(-1)
    assert lib.mla_last_cuda_error(C.byref(err)) == 0 and err.value == 0
    assert lib.mla_last_cuda_error(None) == 1


FAKE = C.c_void_p(0x10000)  # never dereferenced: every call below fails validation first


def decode_call(lib, **over):
    a = dict(q_nope=FAKE, q_rope=FAKE, pool=FAKE, stride=64 * 352, num_blocks=10, bt=FAKE, max_blocks=4, cl=FAKE,
             idx=FAKE, batch=2, heads=16, bs=64, topk=2048, scale=0.07, out=FAKE, lse=None, ws=None, ws_bytes=0)
    a.update(over)
    return lib.mla_sparse_decode(a["q_nope"], a["q_rope"], a["pool"], a["stride"], a["num_blocks"], a["bt"],
                                 a["max_blocks"], a["cl"], a["idx"], a["batch"], a["heads"], a["bs"], a["topk"],
                                 a["scale"], a["out"], a["lse"], a["ws"], a["ws_bytes"], None)


def test_decode_validation(lib):
    INVALID, UNSUPPORTED = 1, 2
    assert decode_call(lib, q_nope=None) == INVALID
    assert decode_call(lib, out=None) == INVALID
    assert decode_call(lib, bs=32) == UNSUPPORTED
    assert decode_call(lib, bs=48) == INVALID
    assert decode_call(lib, heads=8) == INVALID
    assert decode_call(lib, heads=24) == INVALID
    assert decode_call(lib, heads=144) == INVALID
    assert decode_call(lib, topk=0) == INVALID
    assert decode_call(lib, topk=2049) == INVALID
    assert decode_call(lib, scale=float("nan")) == INVALID
    assert decode_call(lib, stride=64 * 352 - 16) == INVALID
    assert decode_call(lib, stride=64 * 352 + 8) == INVALID
    assert decode_call(lib, pool=C.c_void_p(0x10008)) == INVALID  # pool not 16-byte aligned
    assert decode_call(lib, batch=-1) == INVALID
    assert decode_call(lib, max_blocks=0) == INVALID
    assert decode_call(lib, batch=0, q_nope=None) == 0  # empty batch is a no-op


def test_quantize_append_validation(lib):
    f = lib.mla_kv_quantize_append
    assert f(FAKE, FAKE, FAKE, 10, FAKE, 4, 64, 64 * 352, 2, None) == 1        # bad format
    assert f(FAKE, FAKE, FAKE, 10, FAKE, 4, 64, 64 * 352 - 16, 0, None) == 1   # stride too small
    assert f(FAKE, FAKE, FAKE, 10, FAKE, 4, 64, 64 * 576 - 16, 1, None) == 1
    assert f(FAKE, FAKE, FAKE, 10, FAKE, 4, 128, 128 * 352, 0, None) == 2      # block size unsupported
    assert f(None, FAKE, FAKE, 10, FAKE, 4, 64, 64 * 352, 0, None) == 1
    assert f(C.c_void_p(0x10004), FAKE, FAKE, 10, FAKE, 4, 64, 64 * 352, 0, None) == 1  # latent misaligned
    assert f(None, None, None, 0, None, 4, 64, 64 * 352, 0, None) == 0         # n_tokens == 0 is a no-op
    assert f(FAKE, FAKE, FAKE, -1, FAKE, 4, 64, 64 * 352, 0, None) == 1


def test_topk_and_indexer_validation(lib):
    assert lib.mla_topk(FAKE, 100, FAKE, 2, 0, 100, FAKE, None, 0, None) == 1
    assert lib.mla_topk(FAKE, 100, FAKE, 2, 2049, 100, FAKE, None, 0, None) == 1
    assert lib.mla_topk(FAKE, 99, FAKE, 2, 16, 100, FAKE, None, 0, None) == 1   # stride < max_context_len
    assert lib.mla_topk(None, 100, FAKE, 2, 16, 100, FAKE, None, 0, None) == 1
    assert lib.mla_topk(None, 100, None, 0, 16, 100, None, None, 0, None) == 0  # empty batch
    f = lib.mla_indexer_topk
    args = [FAKE, FAKE, FAKE, 64 * 132, 10, FAKE, 4, FAKE, 2, 32, 64, 2048, FAKE, None, 4096, None, 0, None]
    bad_heads = list(args)
    bad_heads[9] = 24
    assert f(*bad_heads) == 2
    bad_heads[9] = 7
    assert f(*bad_heads) == 1
    small_stride = list(args)
    small_stride[3] = 64 * 132 - 16
    assert f(*small_stride) == 1
    no_ws = list(args)
    assert f(*no_ws) == 3  # the scores need workspace
    assert lib.mla_indexer_topk_workspace_size(2, 4096, 2048) >= 2 * 4096 * 4


def test_split_workspace_holds_every_partial(lib):
    """Split partials (normalised O in f16 and a float base-2 LSE per split and
    head) live in the workspace, whether the splits merge inside their
    thread-block cluster (up to 8) or in a second kernel."""
    for batch, splits_at_least in [(32, 2), (2, 32)]:
        need = batch * 16 * splits_at_least * (512 * 2 + 4)
        assert lib.mla_sparse_decode_workspace_size(batch, 16, 2048) >= need


def test_decode_plan(lib):
    """The plan query agrees with the workspace query and the merge rule (up
    to 8 splits merge inside their cluster: one kernel)."""
    import sparse_mla_decode_kv_gb300 as m
    for batch, heads, topk in [(32, 16, 2048), (2, 16, 2048), (1, 16, 1), (128, 64, 2048), (3, 32, 300)]:
        p = m.mla_sparse_decode_plan(batch, heads, topk)
        assert p["rows_per_split"] % 16 == 0 and p["splits"] * p["rows_per_split"] >= topk
        assert (p["splits"] - 1) * p["rows_per_split"] < topk  # no empty split
        assert p["kernels"] == (2 if p["splits"] > 8 else 1)
        assert (lib.mla_sparse_decode_workspace_size(batch, heads, topk) > 0) == (p["splits"] > 1)
    assert lib.mla_sparse_decode_plan(0, 16, 2048, None, None, None) == 1
    assert lib.mla_sparse_decode_plan(4, 8, 2048, None, None, None) == 1
    assert lib.mla_sparse_decode_plan(4, 16, 0, None, None, None) == 1
    assert lib.mla_sparse_decode_plan(4, 16, 2048, None, None, None) == 0


def test_decode_plan_for_format_and_pool(lib):
    """The format-aware plan says when the tensor-memory kernel runs (NVFP4,
    64-head blocks, a pool stride of whole 352-byte rows) and then splits a
    list at most as many ways as the 16-head plan, so its partials fit the
    same workspace."""
    import sparse_mla_decode_kv_gb300 as m
    nvfp4, fp8 = 0, 1
    packed = 64 * 352
    # The kernel also needs the driver's tensor-map encoder: without a driver
    # (a build box) the plan is the 16-head one, as the dispatch would be.
    try:
        C.CDLL("libcuda.so.1")
        driver = True
    except OSError:
        driver = False
    for batch, heads, topk in [(128, 64, 2048), (1, 64, 2048), (2, 128, 700), (6, 64, 2048), (3, 64, 1)]:
        p = m.mla_sparse_decode_plan_fmt(nvfp4, batch, heads, topk, packed, 1000)
        base = m.mla_sparse_decode_plan(batch, heads, topk)
        assert p["tensor_memory"] == driver
        if not driver:
            assert {k: p[k] for k in base} == base
            continue
        assert 1 <= p["splits"] <= base["splits"]
        assert p["splits"] * p["rows_per_split"] >= topk and (p["splits"] - 1) * p["rows_per_split"] < topk
        assert p["kernels"] == (2 if p["splits"] > 1 else 1)
    # everything else is the 16-head plan
    for fmt, heads, stride, nb in [(nvfp4, 16, packed, 1000), (nvfp4, 48, packed, 1000), (fp8, 64, 64 * 576, 1000),
                                   (nvfp4, 64, packed + 16, 1000), (nvfp4, 64, packed, 0)]:
        p = m.mla_sparse_decode_plan_fmt(fmt, 4, heads, 2048, stride, nb)
        base = m.mla_sparse_decode_plan(4, heads, 2048)
        assert not p["tensor_memory"]
        assert {k: p[k] for k in base} == base
    assert lib.mla_sparse_decode_plan_fmt(2, 4, 64, 2048, packed, 10, None, None, None, None) == 1  # unknown fmt
    assert lib.mla_sparse_decode_plan_fmt(0, 4, 8, 2048, packed, 10, None, None, None, None) == 1


def test_workspace_sizes_are_zero_for_empty_or_invalid(lib):
    assert lib.mla_sparse_decode_workspace_size(0, 16, 2048) == 0
    assert lib.mla_sparse_decode_workspace_size(4, 8, 2048) == 0
    assert lib.mla_topk_workspace_size(0, 10, 10) == 0


def test_index_key_append_validation(lib):
    f = lib.mla_index_key_quantize_append
    assert f(FAKE, FAKE, 10, FAKE, 4, 64, 64 * 132 - 16, None) == 1   # stride too small
    assert f(FAKE, FAKE, 10, FAKE, 4, 64, 64 * 132 + 8, None) == 1    # stride not a multiple of 16
    assert f(FAKE, FAKE, 10, FAKE, 4, 32, 32 * 132, None) == 2        # block size unsupported
    assert f(None, FAKE, 10, FAKE, 4, 64, 64 * 132, None) == 1
    assert f(C.c_void_p(0x10008), FAKE, 10, FAKE, 4, 64, 64 * 132, None) == 1  # keys misaligned
    assert f(None, None, 0, None, 4, 64, 64 * 132, None) == 0         # n_tokens == 0 is a no-op
    assert f(FAKE, FAKE, -2, FAKE, 4, 64, 64 * 132, None) == 1


def test_staged_path_validation_and_sizes(lib):
    assert lib.mla_staged_pool_bytes(3, 70) == 3 * 2 * 64 * 576
    assert lib.mla_staged_pool_bytes(0, 70) == 0
    f = lib.mla_stage_rows_fp8
    args = [FAKE, 64 * 352, 10, FAKE, 4, FAKE, FAKE, 2, 64, 2048, FAKE, FAKE, None]
    for i, v, want in [(0, None, 1), (10, None, 1), (11, None, 1), (1, 64 * 352 - 16, 1), (8, 32, 2),
                       (9, 0, 1), (9, 2049, 1), (10, C.c_void_p(0x10008), 1), (4, 0, 1)]:
        a = list(args)
        a[i] = v
        assert f(*a) == want, (i, v)
    empty = list(args)
    empty[7] = 0
    empty[0] = None
    assert f(*empty) == 0
    # the staged decode validates like mla_sparse_decode, then wants its workspace
    need = lib.mla_sparse_decode_staged_workspace_size(2, 16, 2048)
    assert need >= lib.mla_staged_pool_bytes(2, 2048) + 2 * 2048 * 4
    g = lib.mla_sparse_decode_staged
    base = [FAKE, FAKE, FAKE, 64 * 352, 10, FAKE, 4, FAKE, FAKE, 2, 16, 64, 2048, 0.07, FAKE, None, None, 0, None]
    assert g(*base) == 3
    bad = list(base)
    bad[10] = 24
    assert g(*bad) == 1
    bad = list(base)
    bad[3] = 64 * 352 - 16  # stride too small for 352-byte rows
    assert g(*bad) == 1


def test_no_alloc_decode_rejects_scratch_beyond_its_array(lib):
    """mla_sparse_decode_noalloc keeps its split-K scratch in a fixed 16 MiB
    array: a shape whose scratch exceeds it is refused with
    MLA_ERR_WORKSPACE_TOO_SMALL before any device lookup or launch, so the
    call is safe to make on a machine without a GPU."""
    cap = 16 << 20
    f = lib.mla_sparse_decode_noalloc
    for batch, heads in [(128, 128), (512, 16), (128, 64)]:
        need = lib.mla_sparse_decode_workspace_size(batch, heads, 2048)
        assert need > cap, (batch, heads, need)
        assert f(FAKE, FAKE, FAKE, 64 * 352, 10, FAKE, 4, FAKE, FAKE, batch, heads, 64, 2048, 0.07, FAKE, None,
                 None) == 3
    assert 0 < lib.mla_sparse_decode_workspace_size(32, 16, 2048) <= cap  # the TP4 rank fits
