"""The C-ABI library builds, loads, and exports every symbol its header declares (CPU only)."""
import ctypes
import os
import re

import pytest

import paged_sparse_mla_gb300 as smla
from paged_sparse_mla_gb300 import build_lib
import oracle

HEADER = os.path.join(build_lib.ROOT, "include", "smla.h")


@pytest.fixture(scope="module")
def lib():
    build_lib.build()
    return smla.lib()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", text, flags=re.M)) - {"if"}


def test_every_declared_symbol_is_exported(lib):
    declared = _declared()
    assert declared == set(smla.EXPORTED_SYMBOLS), declared ^ set(smla.EXPORTED_SYMBOLS)
    for name in declared:
        assert hasattr(lib, name), name


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
def test_layout_init_matches_oracle_layout(lib, fmt):
    for args in [(64, 1, 512, 64, 128, 128, 1000), (16, 1, 64, 16, 64, 32, 32), (64, 3, 512, 64, 128, 128, 7)]:
        lay = smla.layout_init(*args, key_format=fmt)
        ref = oracle.PoolLayout(*args, fmt)
        assert lay.key_bytes == ref.key_bytes and lay.idx_key_format == smla.KEY_FORMATS[fmt]
        assert lay.rec_stride == ref.rec_stride and lay.rec_bytes == ref.rec_bytes
        assert lay.idx_key_off == ref.idx_key_off and lay.idx_scale_off == ref.idx_scale_off
        assert lay.layer_stride == ref.layer_stride and lay.block_stride == ref.block_stride
        assert lay.pool_bytes == ref.pool_bytes


@pytest.mark.parametrize("bad", [(0, 1, 512, 64, 128, 128, 10), (64, 1, 500, 64, 128, 128, 10),
                                 (64, 1, 512, 64, 100, 128, 10), (64, 1, 512, 63, 128, 128, 10),
                                 (64, 1, 512, 64, 128, 120, 10), (64, 0, 512, 64, 128, 128, 10)])
def test_layout_init_rejects_bad_shapes(lib, bad):
    with pytest.raises(smla.SmlaError) as e:
        smla.layout_init(*bad)
    assert e.value.code == 1


def test_fp4_key_layout_and_its_refusals(lib):
    """smla_layout_init_keys: E2M1 keys halve the key region; unknown formats and d_index not a multiple
    of 32 are refused; an E2M1 layout with a shape the FP4 indexer is not built for is UNSUPPORTED before
    any device work."""
    lay = smla.layout_init(64, 1, 512, 64, 128, 128, 10, key_format="e2m1")
    assert (lay.idx_key_off, lay.idx_scale_off, lay.block_stride) == (41984, 46080, 46336)
    L = ctypes.byref(smla.Layout())
    assert lib.smla_layout_init_keys(L, 64, 1, 512, 64, 128, 128, 2, 10) == 1      # unknown format
    assert lib.smla_layout_init_keys(L, 64, 1, 512, 64, 128, 48, 1, 10) == 1       # d_index % 32 != 0
    assert lib.smla_layout_init_keys(L, 64, 1, 512, 64, 128, 48, 0, 10) == 0       # fine as E4M3
    tiny = smla.layout_init(16, 1, 64, 16, 64, 32, 32, key_format="e2m1")
    prm = smla.make_params(8, 4, 64, 0.1)
    p = ctypes.c_void_p(4096)
    step = (p, 0, p, p, p, p, p, p, p, p, p, p, 16, p, p, 1, 1, 1, 100, p, p, None)
    assert lib.smla_decode(ctypes.byref(tiny), ctypes.byref(prm), *step, p, 1 << 30, None) == 2
    assert lib.smla_decode_static(ctypes.byref(tiny), ctypes.byref(prm), *step, None) == 2


def test_host_side_argument_checks(lib):
    lay = smla.layout_init(64, 1, 512, 64, 128, 128, 10)
    prm = smla.make_params(64, 64, 2048, 1 / 24)
    L = ctypes.byref(lay)
    P = ctypes.byref(prm)
    # null descriptors / pointers are rejected before any device work
    assert lib.kvpack_store(None, None, 0, None, None, None, None, None, 1, None) == 1
    assert lib.kvpack_store(L, None, 0, None, None, None, None, None, 1, None) == 1
    assert lib.kvpack_store(L, None, 0, None, None, None, None, None, 0, None) == 0   # nothing to do
    assert lib.kvpack_store(L, ctypes.c_void_p(256), 5, None, None, None, None, None, 1, None) == 1  # bad layer
    assert lib.smla_topk(P, None, 0, None, None, 1, 4, None, None, 0, None) == 1
    assert lib.smla_topk_workspace_size(P, 4) > 0               # few rows: the segment scratch
    assert lib.smla_topk_workspace_size(P, 100000) == 0         # many rows: no split
    assert lib.smla_attend(L, P, None, 0, None, None, None, None, 0, None, 1, 3, None, None, None, 0, None) == 1
    # a workspace size without a workspace is an argument error
    assert lib.smla_attend(L, P, None, 0, None, None, None, None, 0, None, 1, 0, None, None, None, 64, None) == 1
    assert lib.smla_attend_workspace_size(L, P, 4) > 0          # few tokens: the split scratch
    assert lib.smla_attend_workspace_size(L, P, 100000) == 0    # many tokens: no split
    assert lib.smla_decode(L, P, None, 0, None, None, None, None, None, None, None, None, None, None, 0, None,
                           None, 1, 4, 1, 100, None, None, None, None, 0, None) == 1
    # prefill chunks must store their own keys first: no slot mapping is an argument error
    assert lib.smla_prefill_chunk(L, P, None, 0, None, None, None, None, None, None, None, None, None, None, 0, None,
                                  None, 1, 4, 4, 100, None, None, None, None, 0, None) == 1
    assert lib.smla_prefill_chunk(L, P, None, 0, None, None, None, None, None, None, None, None, None, None, 0, None,
                                  None, 1, 0, 4, 100, None, None, None, None, 0, None) == 0  # an empty chunk
    assert lib.smla_workspace_size(L, P, 0, 100) == 0
    assert lib.smla_workspace_size(L, P, 4, 1000) >= 4 * 1000 * 4 + 4 * 2048 * 4
    assert lib.smla_selftest_wait(0, None) == 1                  # wait limit below 1 ms
    assert lib.smla_selftest_wait(20_000_000_000, None) == 1     # above 10 s
    assert lib.smla_status_string(4) == b"SMLA_ERR_BAD_INDEX"
    assert lib.smla_version() >= 100


@pytest.mark.parametrize("field,delta", [("idx_key_off", 16), ("block_stride", -256), ("rec_stride", 16),
                                         ("quant_tile", -128), ("layer_stride", 256), ("n_scales", 1),
                                         ("idx_key_format", 1)])
def test_layouts_not_made_by_layout_init_are_refused_everywhere(lib, field, delta):
    """Every entry point that takes a layout refuses one whose fields differ from smla_layout_init's,
    before any device work; the two fused entry points answer alike."""
    lay = smla.layout_init(64, 1, 512, 64, 128, 128, 10)
    setattr(lay, field, getattr(lay, field) + delta)
    prm = smla.make_params(64, 64, 2048, 1 / 24)
    L, P = ctypes.byref(lay), ctypes.byref(prm)
    p = ctypes.c_void_p(4096)                                    # never dereferenced on the host
    assert lib.smla_workspace_size(L, P, 4, 1000) == 0
    assert lib.smla_attend_workspace_size(L, P, 4) == 0
    assert lib.kvpack_store(L, p, 0, p, p, p, p, p, 1, None) == 1
    assert lib.smla_index_scores(L, P, p, 0, p, p, p, 16, p, p, 1, 1, 1, 1000, p, 1000, None) == 1
    assert lib.smla_attend(L, P, p, 0, p, p, p, p, 16, p, 1, 1, p, p, None, 0, None) == 1
    step = (p, 0, p, p, p, p, p, p, p, p, p, p, 16, p, p, 1, 1, 1, 1000, p, p, None)
    assert lib.smla_decode(L, P, *step, p, 1 << 30, None) == 1
    assert lib.smla_decode_static(L, P, *step, None) == 1


@pytest.mark.parametrize("case", ["q_pe", "n_heads", "n_idx_heads", "top_k", "unbuilt_idx_heads", "unbuilt_heads"])
def test_fused_entry_points_refuse_the_same_arguments(lib, case):
    """smla_decode and smla_decode_static apply the same checks and return the same status, with
    nothing enqueued (these run without a GPU)."""
    lay = smla.layout_init(64, 1, 512, 64, 128, 128, 10)
    prm = smla.make_params(64, 64, 2048, 1 / 24)
    p = ctypes.c_void_p(4096)
    q_pe = None if case == "q_pe" else p
    want = 1
    if case in ("n_heads", "n_idx_heads", "top_k"):
        setattr(prm, case, 0)
    if case == "unbuilt_idx_heads":
        prm.n_idx_heads, want = 32, 2
    if case == "unbuilt_heads":
        prm.n_heads, want = 65, 2
    L, P = ctypes.byref(lay), ctypes.byref(prm)
    step = (p, 0, p, p, p, p, p, p, q_pe, p, p, p, 16, p, p, 1, 1, 1, 1000, p, p, None)
    a = lib.smla_decode(L, P, *step, p, 1 << 30, None)
    b = lib.smla_decode_static(L, P, *step, None)
    assert a == b == want


def test_header_is_c99_and_the_library_links_from_c(lib, tmp_path):
    """A plain C caller (tests/c/abi_host_check.c) compiles against include/smla.h with gcc -std=c99
    -pedantic -Werror, links libsmla.so and gets the documented host-side answers."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = os.path.join(build_lib.ROOT, "tests", "c", "abi_host_check.c")
    exe = str(tmp_path / "abi_host_check")
    lib_dir = os.path.dirname(build_lib.LIB)
    cc = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I",
                         os.path.dirname(HEADER), src, "-L", lib_dir, "-lsmla", f"-Wl,-rpath,{lib_dir}", "-o", exe],
                        capture_output=True, text=True)
    assert cc.returncode == 0, cc.stderr
    run = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, run.stderr
    assert "abi host check ok" in run.stdout
