"""The C-ABI library loads, exports every symbol include/dcpmla.h declares, and rejects
invalid arguments on the host before any launch (these calls touch no GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dcpmla.h")


@pytest.fixture(scope="module")
def lib():
    from decode_context_sparse_gb300 import build
    build.build()
    import decode_context_sparse_gb300 as dcp
    return dcp.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(",
                       src, flags=re.M)
    return sorted(set(n for n in names if not n.startswith("defined")))


def test_header_declares_the_four_path_entry_points():
    names = declared_functions()
    for n in ("dcp_remap_topk", "mla_decode_partial_lse", "dcp_lse_merge", "mla_decode_dcp_fused"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    import decode_context_sparse_gb300 as dcp
    names = declared_functions()
    assert sorted(dcp.EXPORTS) == names
    for n in names:
        assert hasattr(lib, n), n


def test_abi_version_and_status_strings(lib):
    import decode_context_sparse_gb300 as dcp
    assert lib.dcp_abi_version() == dcp.DCP_ABI_VERSION
    for st in (0, -1, -2, -3, -4):
        assert lib.dcp_status_string(st).decode().startswith("DCP_")
    assert b"unknown" in lib.dcp_status_string(7)


def test_remap_rejects_bad_arguments(lib):
    good = ctypes.c_void_p(256)
    call = lib.dcp_remap_topk
    assert call(None, 4, 8, 2, 1, -1, good, good, None) == -1          # null input
    assert call(good, 4, 0, 2, 1, -1, good, good, None) == -1          # k < 1
    assert call(good, 4, 1 << 20, 2, 1, -1, good, good, None) == -1    # k too large
    assert call(good, 4, 8, 0, 1, -1, good, good, None) == -1          # dcp < 1
    assert call(good, 4, 8, 65, 1, -1, good, good, None) == -1         # dcp too large
    assert call(good, 4, 8, 2, 0, -1, good, good, None) == -1          # interleave < 1
    assert call(good, 4, 8, 2, 1, 2, good, good, None) == -1           # shard >= dcp
    assert call(good, -1, 8, 2, 1, -1, good, good, None) == -1         # rows < 0


def test_merge_rejects_bad_arguments(lib):
    g = ctypes.c_void_p(4096)
    call = lib.dcp_lse_merge
    assert call(None, g, 2, 4, 8, 512, g, g, None) == -1
    assert call(g, g, 0, 4, 8, 512, g, g, None) == -1
    assert call(g, g, 2, 4, 8, 510, g, g, None) == -1                  # dv % 4
    assert call(ctypes.c_void_p(4100), g, 2, 4, 8, 512, g, g, None) == -1  # misaligned


def _args(**kw):
    import decode_context_sparse_gb300 as dcp
    a = dcp.DecodeArgs()
    p = 1 << 20
    a.q = p; a.rows = 4; a.heads = 128; a.sm_scale = 0.07
    a.kv_pool = p; a.num_pages = 10; a.kv_dtype = 1; a.page_size = 64
    a.block_table = p; a.num_seqs = 2; a.bt_stride = 4; a.row_seq = p
    a.idx = p; a.count = p; a.k = 2048
    a.out = p; a.lse = p
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def test_decode_rejects_bad_arguments(lib):
    import decode_context_sparse_gb300 as dcp
    part, fused = lib.mla_decode_partial_lse, lib.mla_decode_dcp_fused
    R = ctypes.byref
    assert part(R(_args(q=None)), 1, None) == dcp.DCP_ERR_INVALID_ARG
    assert part(R(_args(q=(1 << 20) + 2)), 1, None) == dcp.DCP_ERR_INVALID_ARG   # misaligned q
    assert part(R(_args(heads=100)), 1, None) == dcp.DCP_ERR_UNSUPPORTED
    assert part(R(_args(heads=256)), 1, None) == dcp.DCP_ERR_UNSUPPORTED
    assert part(R(_args(page_size=16)), 1, None) == dcp.DCP_ERR_UNSUPPORTED
    assert part(R(_args(kv_dtype=5)), 1, None) == dcp.DCP_ERR_UNSUPPORTED
    assert part(R(_args(k=0)), 1, None) == dcp.DCP_ERR_INVALID_ARG
    assert part(R(_args(count=None)), 1, None) == dcp.DCP_ERR_INVALID_ARG      # sparse partial
    assert part(R(_args()), 0, None) == dcp.DCP_ERR_INVALID_ARG                # no shards
    assert part(R(_args(idx=None)), 1, None) == dcp.DCP_ERR_INVALID_ARG        # dense w/o kv_len
    assert fused(R(_args()), 0, 1, None) == dcp.DCP_ERR_INVALID_ARG
    assert fused(R(_args()), 8, 0, None) == dcp.DCP_ERR_INVALID_ARG
    # a split-KV call without workspace is refused before launch
    assert fused(R(_args(num_splits=4)), 8, 1, None) == dcp.DCP_ERR_WORKSPACE
    assert lib.mla_decode_workspace_size(R(_args(num_splits=4)), 8, 1) > 0
    assert lib.mla_decode_workspace_size(R(_args(q=None)), 8, 1) == ctypes.c_size_t(-1).value
    # the CUDA-core path (up to 32 heads) needs none without splits; the tensor-core path
    # (48..128 heads) always reserves its split-unit partials and tickets
    assert lib.mla_decode_workspace_size(R(_args(num_splits=1, heads=32)), 8, 1) == 0
    assert lib.mla_decode_workspace_size(R(_args(num_splits=1)), 8, 1) > 0


def test_kv_cache_write_rejects_bad_arguments(lib):
    import decode_context_sparse_gb300 as dcp
    g = ctypes.c_void_p(1 << 20)
    call = lib.dcp_kv_cache_write
    ok = dict(kv=g, n=4, seq=g, pos=g, dcp=2, interleave=1, shard=-1, pool=g, num_pages=8,
              kv_dtype=1, page_size=64, bt=g, num_seqs=1, bt_stride=4, checked=0, err=None)

    def run(**kw):
        a = dict(ok, **kw)
        return call(a["kv"], a["n"], a["seq"], a["pos"], a["dcp"], a["interleave"], a["shard"],
                    a["pool"], a["num_pages"], a["kv_dtype"], a["page_size"], a["bt"],
                    a["num_seqs"], a["bt_stride"], a["checked"], a["err"], None)
    assert run(kv=None) == dcp.DCP_ERR_INVALID_ARG
    assert run(pool=None) == dcp.DCP_ERR_INVALID_ARG
    assert run(kv=ctypes.c_void_p((1 << 20) + 8)) == dcp.DCP_ERR_INVALID_ARG   # misaligned rows
    assert run(n=-1) == dcp.DCP_ERR_INVALID_ARG
    assert run(dcp=0) == dcp.DCP_ERR_INVALID_ARG
    assert run(shard=2) == dcp.DCP_ERR_INVALID_ARG
    assert run(num_pages=0) == dcp.DCP_ERR_INVALID_ARG
    assert run(page_size=32) == dcp.DCP_ERR_UNSUPPORTED
    assert run(kv_dtype=3) == dcp.DCP_ERR_UNSUPPORTED
    assert run(n=0) == dcp.DCP_OK    # nothing to do, nothing launched


def test_topk_entries_reject_bad_arguments(lib):
    import decode_context_sparse_gb300 as dcp
    g = ctypes.c_void_p(1 << 20)
    bad = ctypes.c_void_p((1 << 20) + 2)
    loc = lib.dcp_topk_local
    ok = dict(sc=g, rows=4, stride=1000, ln=g, k=16, dcp=2, il=1, shard=-1, cs=g, ci=g)

    def run_l(**kw):
        a = dict(ok, **kw)
        return loc(a["sc"], a["rows"], a["stride"], a["ln"], a["k"], a["dcp"], a["il"], a["shard"],
                   a["cs"], a["ci"], None)
    E = dcp.DCP_ERR_INVALID_ARG
    assert run_l(sc=None) == E
    assert run_l(ci=None) == E
    assert run_l(sc=bad) == E                       # misaligned scores
    assert run_l(rows=-1) == E
    assert run_l(stride=0) == E
    assert run_l(k=0) == E and run_l(k=dcp.DCP_MAX_TOPK + 1) == E
    assert run_l(dcp=0) == E and run_l(shard=2) == E and run_l(il=0) == E
    assert run_l(stride=1 << 30, dcp=8) == E        # global slot ids past INT32_MAX
    assert run_l(rows=0) == dcp.DCP_OK              # nothing to do, nothing launched
    mrg = lib.dcp_topk_merge
    okm = dict(cs=g, ci=g, dcp=8, rows=4, kin=2048, k=2048, top=g, cnt=g)

    def run_m(**kw):
        a = dict(okm, **kw)
        return mrg(a["cs"], a["ci"], a["dcp"], a["rows"], a["kin"], a["k"], a["top"], a["cnt"], None)
    assert run_m(cs=None) == E and run_m(top=None) == E
    assert run_m(dcp=0) == E and run_m(dcp=dcp.DCP_MAX_SHARDS + 1) == E
    assert run_m(rows=-1) == E and run_m(kin=0) == E and run_m(k=0) == E
    assert run_m(k=dcp.DCP_MAX_TOPK + 1) == E
    assert run_m(dcp=64, kin=1 << 26) == E          # D * k_in past INT32_MAX
    assert run_m(top=bad) == E
    assert run_m(rows=0) == dcp.DCP_OK


def test_prefill_chunk_entry_checks(lib):
    import decode_context_sparse_gb300 as dcp
    R = ctypes.byref
    E = dcp.DCP_ERR_INVALID_ARG
    good = dict(kv_len=1 << 20, max_kv_len=5000)
    assert lib.mla_prefill_chunk_workspace_size(R(_args(**good)), 8, 1) > 0
    assert lib.mla_prefill_chunk_workspace_size(R(_args(idx=None, **good)), 8, 1) == \
        ctypes.c_size_t(-1).value
    assert lib.mla_prefill_chunk_dcp(None, 8, 1, None) == E
    assert lib.mla_prefill_chunk_dcp(R(_args(**good)), 8, 1, None) == dcp.DCP_ERR_WORKSPACE
    assert lib.mla_prefill_chunk_dcp(R(_args(**good)), 33, 1, None) == dcp.DCP_ERR_UNSUPPORTED
    assert lib.mla_prefill_chunk_dcp(R(_args(max_kv_len=5000)), 8, 1, None) == E   # no prefix lengths
    assert lib.mla_prefill_chunk_dcp(R(_args(idx=None, **good)), 8, 1, None) == E   # no chunk slots
    assert lib.mla_prefill_chunk_dcp(R(_args(**good)), 8, 0, None) == E            # interleave 0


def test_kernel_path_field(lib):
    import decode_context_sparse_gb300 as dcp
    R = ctypes.byref
    # an unknown kernel choice is refused before any launch
    assert lib.mla_decode_dcp_fused(R(_args(kernel_path=7)), 8, 1, None) == dcp.DCP_ERR_INVALID_ARG
    assert lib.mla_decode_workspace_size(R(_args(kernel_path=-1)), 8, 1) == ctypes.c_size_t(-1).value
    # the field is read: with 128 heads and one split the CUDA-core kernel needs no workspace,
    # the tensor-core kernel (the automatic choice) does
    assert lib.mla_decode_workspace_size(R(_args(num_splits=1, kernel_path=dcp.DCP_PATH_CUDA_CORES)),
                                         8, 1) == 0
    assert lib.mla_decode_workspace_size(R(_args(num_splits=1, kernel_path=dcp.DCP_PATH_AUTO)),
                                         8, 1) > 0


def test_args_struct_layout_matches_header(tmp_path):
    """The binding's ctypes mirror of dcp_mla_decode_args has the C compiler's layout: a tiny C
    program built against include/dcpmla.h prints every field's offset and the size."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    import decode_context_sparse_gb300 as dcp
    names = [f[0] for f in dcp.DecodeArgs._fields_]
    src = tmp_path / "layout.c"
    body = "".join('  printf("%%s %%zu\\n", "%s", offsetof(dcp_mla_decode_args, %s));\n' % (n, n)
                   for n in names)
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "dcpmla.h"\nint main(void) {\n'
                   + body + '  printf("sizeof %zu\\n", sizeof(dcp_mla_decode_args));\n  return 0;\n}\n')
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)])
    got = dict(line.split() for line in subprocess.check_output([str(exe)]).decode().splitlines())
    for n in names:
        assert int(got[n]) == getattr(dcp.DecodeArgs, n).offset, n
    assert int(got["sizeof"]) == ctypes.sizeof(dcp.DecodeArgs)
