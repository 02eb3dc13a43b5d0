"""The oracle -- TEST INFRASTRUCTURE ONLY.

A plain double-precision CPU statement of the decode-context-parallel (DCP) MLA decode
path, used to check the CUDA library.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import it.  The product package never imports
it and shares no code with it; the C source is ``oracle/dcp_oracle.c`` and is built with
gcc (OpenMP) by :func:`build`.

Functions (each follows a passage of the public pages on DCP, cited in the C source):
  * :func:`e4m3_decode`   -- the E4M3 format definition, all 256 codes;
  * :func:`owner`, :func:`local` -- the owner rule and local slot id (reading stated in C);
  * :func:`count_owned`   -- brute-force count of a shard's slots below a length;
  * :func:`remap`         -- top-k slot remap per shard (stable compaction + count);
  * :func:`attention`     -- sparse or dense MLA decode attention with LSE, unsharded or
    restricted to one shard, brute force over the selected slots;
  * :func:`merge`         -- LSE merge of shard partials with the all-empty case;
  * :func:`e4m3_encode`, :func:`kv_write` -- FP8 quantisation and the DCP KV-cache write;
  * ``oracle.topk``        -- the DSA top-k producer under DCP (per-shard candidates and
    their merge; numpy, see that module).

Parity status: every function above is pinned against closed forms, hand-worked fixtures
(``tests/golden/``), brute-force enumeration and invariants by ``tests/test_oracle_pins.py``,
``tests/test_oracle_kv_write_pins.py`` and ``tests/test_oracle_topk_pins.py``; none is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dcp_oracle.c")
_SO = os.path.join(_HERE, "_dcp_oracle.so")
_lib = None

KV_BF16 = 0
KV_FP8 = 1


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc -O2 -fopenmp into oracle/_dcp_oracle.so."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + ".tmp%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp", _SRC, "-o", tmp, "-lm"]
        subprocess.check_call(cmd)
        os.replace(tmp, _SO)
    return _SO


class _AttnArgs(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("rows", ctypes.c_int64), ("heads", ctypes.c_int32),
        ("sm_scale", ctypes.c_double), ("pool", ctypes.c_void_p), ("num_pages", ctypes.c_int64),
        ("kv_dtype", ctypes.c_int32), ("page_size", ctypes.c_int32),
        ("block_table", ctypes.c_void_p), ("num_seqs", ctypes.c_int32),
        ("bt_stride", ctypes.c_int32), ("row_seq", ctypes.c_void_p),
        ("row_len", ctypes.c_void_p), ("topk", ctypes.c_void_p), ("k", ctypes.c_int32),
        ("dcp", ctypes.c_int32), ("interleave", ctypes.c_int32), ("shard", ctypes.c_int32),
        ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p),
    ]


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.orc_e4m3_decode.restype = ctypes.c_double
        lib.orc_e4m3_decode.argtypes = [ctypes.c_int]
        lib.orc_owner.restype = ctypes.c_int
        lib.orc_owner.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_int]
        lib.orc_local.restype = ctypes.c_int64
        lib.orc_local.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_int]
        lib.orc_count_owned.restype = ctypes.c_int64
        lib.orc_count_owned.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        lib.orc_remap.restype = ctypes.c_int
        lib.orc_remap.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                  ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
        lib.orc_attention.restype = ctypes.c_int
        lib.orc_attention.argtypes = [ctypes.POINTER(_AttnArgs)]
        lib.orc_merge.restype = ctypes.c_int
        lib.orc_merge.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                  ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
        lib.orc_num_threads.restype = ctypes.c_int
        lib.orc_e4m3_encode.restype = ctypes.c_int
        lib.orc_e4m3_encode.argtypes = [ctypes.c_float]
        lib.orc_kv_write.restype = ctypes.c_int64
        lib.orc_kv_write.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                     ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                                     ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                                     ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p]
        _lib = lib
    return _lib


def num_threads() -> int:
    return _load().orc_num_threads()


def _np(x, dtype):
    """Host numpy array (C-contiguous) from a numpy array or torch tensor.

    dtype=np.uint8 reinterprets the raw bytes (bf16 / fp8 tensors); any other dtype
    converts values."""
    if hasattr(x, "detach"):
        import torch
        x = x.detach().cpu().contiguous()
        if x.dtype == torch.bfloat16:
            x = x.view(torch.int16)
        elif x.dtype == torch.float8_e4m3fn:
            x = x.view(torch.uint8)
        x = x.numpy()
    x = np.ascontiguousarray(x)
    if x.dtype != dtype:
        x = x.view(np.uint8) if dtype == np.uint8 else x.astype(dtype)
    return np.ascontiguousarray(x)


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def e4m3_decode(code: int) -> float:
    return _load().orc_e4m3_decode(int(code))


def e4m3_table() -> np.ndarray:
    return np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)


def owner(t: int, dcp: int, interleave: int) -> int:
    return _load().orc_owner(int(t), int(dcp), int(interleave))


def local(t: int, dcp: int, interleave: int) -> int:
    return _load().orc_local(int(t), int(dcp), int(interleave))


def count_owned(length: int, dcp: int, interleave: int, shard: int) -> int:
    return _load().orc_count_owned(int(length), int(dcp), int(interleave), int(shard))


def remap(gidx, dcp: int, interleave: int, shard: int = -1):
    """Returns (local_idx [n_out, rows, k] int32, count [n_out, rows] int32)."""
    g = _np(gidx, np.int32)
    rows, k = g.shape
    n_out = dcp if shard < 0 else 1
    loc = np.empty((n_out, rows, k), dtype=np.int32)
    cnt = np.empty((n_out, rows), dtype=np.int32)
    rc = _load().orc_remap(_ptr(g), rows, k, dcp, interleave, shard, _ptr(loc), _ptr(cnt))
    if rc != 0:
        raise RuntimeError("oracle remap failed: %d" % rc)
    return loc, cnt


def attention(q, pool, block_table, row_seq, dcp, interleave, kv_dtype, sm_scale,
              topk=None, row_len=None, shard=-1, page_size=64):
    """Sparse (topk given) or dense (row_len given) MLA decode attention with LSE.

    q: [R, H, 576] bf16 (torch tensor or uint16/int16 numpy bits); pool: [pages, page, bytes]
    uint8; block_table [D, B, maxp] int32; row_seq [R]; topk [R, K] global slots.
    Returns (out [R, H, 512] float64, lse [R, H] float64).
    """
    qn = _np(q, np.uint8)
    pn = _np(pool, np.uint8)
    bt = _np(block_table, np.int32)
    rs = _np(row_seq, np.int32)
    R = rs.shape[0]
    H = qn.size // (R * 576 * 2)
    tk = _np(topk, np.int32) if topk is not None else None
    rl = _np(row_len, np.int32) if row_len is not None else None
    out = np.zeros((R, H, 512), dtype=np.float64)
    lse = np.zeros((R, H), dtype=np.float64)
    a = _AttnArgs()
    a.q = qn.ctypes.data
    a.rows = R
    a.heads = H
    a.sm_scale = float(sm_scale)
    a.pool = pn.ctypes.data
    a.num_pages = pn.shape[0]
    a.kv_dtype = int(kv_dtype)
    a.page_size = int(page_size)
    a.block_table = bt.ctypes.data
    a.num_seqs = bt.shape[1]
    a.bt_stride = bt.shape[2]
    a.row_seq = rs.ctypes.data
    a.row_len = rl.ctypes.data if rl is not None else None
    a.topk = tk.ctypes.data if tk is not None else None
    a.k = tk.shape[1] if tk is not None else 0
    a.dcp = int(dcp)
    a.interleave = int(interleave)
    a.shard = int(shard)
    a.out = out.ctypes.data
    a.lse = lse.ctypes.data
    rc = _load().orc_attention(ctypes.byref(a))
    if rc != 0:
        raise RuntimeError("oracle attention failed: %d (out-of-range page or bad args)" % rc)
    return out, lse


def attention_problem(p, rows=None, shard=-1):
    """attention() on a synth.DecodeProblem, optionally on a subset of its rows."""
    import torch
    sel = slice(None) if rows is None else torch.as_tensor(rows, dtype=torch.long)
    q = p.q[sel].cpu()
    rs = p.row_seq[sel].cpu()
    tk = p.topk[sel].cpu() if p.topk is not None else None
    rl = p.row_len[sel].cpu()
    return attention(q, p.pool.cpu() if p.pool.is_cuda else p.pool, p.block_table.cpu(), rs,
                     p.dcp, p.interleave, p.kv_dtype, p.sm_scale, topk=tk, row_len=rl,
                     shard=shard, page_size=p.page_size)


def merge(part_out, part_lse):
    """LSE merge: part_out [D, R, H, dv], part_lse [D, R, H] -> (out [R,H,dv], lse [R,H])."""
    po = _np(part_out, np.float64)
    pl = _np(part_lse, np.float64)
    D, R, H, dv = po.shape
    out = np.empty((R, H, dv), dtype=np.float64)
    lse = np.empty((R, H), dtype=np.float64)
    rc = _load().orc_merge(_ptr(po), _ptr(pl), D, R, H, dv, _ptr(out), _ptr(lse))
    if rc != 0:
        raise RuntimeError("oracle merge failed: %d" % rc)
    return out, lse


def e4m3_encode(y: float) -> int:
    """Nearest E4M3 code of the fp32 value y (ties to even, saturating at 448)."""
    return _load().orc_e4m3_encode(float(y))


def kv_write(kv, seq, pos, pool, kv_dtype: int, block_table, dcp: int, interleave: int,
             shard: int = -1):
    """DCP KV-cache write of token rows kv [n, 576] (bf16) at (seq[i], pos[i]) into a copy of
    pool [num_pages, page_size, token_bytes]; returns (new pool uint8, written, skipped)."""
    kvb = _np(kv, np.uint8).reshape(-1, 1152)
    n = kvb.shape[0]
    seq_a = _np(seq, np.int32).reshape(-1)
    pos_a = _np(pos, np.int32).reshape(-1)
    out = _np(pool, np.uint8).copy()
    num_pages, page_size = out.shape[0], out.shape[1]
    bt = _np(block_table, np.int32)
    skipped = ctypes.c_int64(0)
    written = _load().orc_kv_write(_ptr(kvb), n, _ptr(seq_a), _ptr(pos_a), int(dcp), int(interleave),
                                   int(shard), _ptr(out), num_pages, int(kv_dtype), page_size,
                                   _ptr(bt), bt.shape[1], bt.shape[2], ctypes.byref(skipped))
    return out, int(written), int(skipped.value)


from . import topk  # noqa: E402  (numpy-only; no C build needed)
