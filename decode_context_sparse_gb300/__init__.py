"""GB300-native DCP (decode context parallelism) MLA / DSA decode hot path.

A thin Python binding over the C-ABI library ``libdcpmla.so`` (see ``include/dcpmla.h``).
The functions here carry the same names as the C entry points and only marshal
arguments (torch CUDA tensors -> device pointers, current stream); every step of the
computation runs in the library's CUDA kernels.  There is no CPU fallback: if the
library is missing or no GPU is present the calls raise.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdcpmla.so")

DCP_OK = 0
DCP_ERR_INVALID_ARG = -1
DCP_ERR_UNSUPPORTED = -2
DCP_ERR_CUDA = -3
DCP_ERR_WORKSPACE = -4
DCP_KV_BF16 = 0
DCP_KV_FP8_E4M3_S128 = 1
DCP_ERRBIT_SLOT_RANGE = 1
DCP_ERRBIT_PAGE_RANGE = 2
DCP_ERRBIT_TIMEOUT = 4
DCP_MAX_SHARDS = 64
DCP_MAX_TOPK = 16384
DCP_ABI_VERSION = 2
DCP_PATH_AUTO = 0          # tensor cores for 48..128 heads, CUDA cores otherwise
DCP_PATH_CUDA_CORES = 1    # the CUDA-core kernel for every head count
TOKEN_BYTES = {DCP_KV_BF16: 1152, DCP_KV_FP8_E4M3_S128: 656}

# every symbol include/dcpmla.h declares
EXPORTS = ("dcp_status_string", "dcp_abi_version", "dcp_remap_topk", "dcp_local_lengths",
           "mla_decode_partial_lse", "dcp_lse_merge", "mla_decode_dcp_fused",
           "mla_decode_workspace_size", "mla_decode_dcp_fused_noalloc", "dcp_kv_cache_write",
           "dcp_topk_local", "dcp_topk_merge", "mla_prefill_chunk_workspace_size",
           "mla_prefill_chunk_dcp")
DCP_NOALLOC_SCRATCH_BYTES = 16 << 20


class DcpError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__("%s: %s" % (what, _status_string(status)))
        self.status = status


class DecodeArgs(ctypes.Structure):
    """Mirror of dcp_mla_decode_args."""
    _fields_ = [
        ("q", ctypes.c_void_p), ("rows", ctypes.c_int64), ("heads", ctypes.c_int32),
        ("sm_scale", ctypes.c_float),
        ("kv_pool", ctypes.c_void_p), ("num_pages", ctypes.c_int64), ("kv_dtype", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("block_table", ctypes.c_void_p), ("num_seqs", ctypes.c_int32), ("bt_stride", ctypes.c_int32),
        ("row_seq", ctypes.c_void_p),
        ("idx", ctypes.c_void_p), ("count", ctypes.c_void_p), ("k", ctypes.c_int32),
        ("kv_len", ctypes.c_void_p), ("max_kv_len", ctypes.c_int32),
        ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("num_splits", ctypes.c_int32),
        ("checked", ctypes.c_int32), ("err_flag", ctypes.c_void_p),
        ("kernel_path", ctypes.c_int32),
    ]


_lib = None


def load(path: str = LIB_PATH):
    """Load libdcpmla.so (built by decode_context_sparse_gb300.build.build())."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError("libdcpmla.so not found at %s: run __graft_entry__.build() "
                           "(there is no CPU fallback)" % path)
    lib = ctypes.CDLL(path)
    V, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    lib.dcp_status_string.restype = ctypes.c_char_p
    lib.dcp_status_string.argtypes = [ctypes.c_int]
    lib.dcp_abi_version.restype = ctypes.c_int
    lib.dcp_abi_version.argtypes = []
    lib.dcp_remap_topk.restype = ctypes.c_int
    lib.dcp_remap_topk.argtypes = [V, I64, I32, I32, I32, I32, V, V, V]
    lib.dcp_local_lengths.restype = ctypes.c_int
    lib.dcp_local_lengths.argtypes = [V, I64, I32, I32, I32, V, V]
    lib.mla_decode_partial_lse.restype = ctypes.c_int
    lib.mla_decode_partial_lse.argtypes = [ctypes.POINTER(DecodeArgs), I32, V]
    lib.dcp_lse_merge.restype = ctypes.c_int
    lib.dcp_lse_merge.argtypes = [V, V, I32, I64, I32, I32, V, V, V]
    lib.mla_decode_dcp_fused.restype = ctypes.c_int
    lib.mla_decode_dcp_fused.argtypes = [ctypes.POINTER(DecodeArgs), I32, I32, V]
    lib.mla_decode_dcp_fused_noalloc.restype = ctypes.c_int
    lib.mla_decode_dcp_fused_noalloc.argtypes = [ctypes.POINTER(DecodeArgs), I32, I32, V]
    lib.dcp_kv_cache_write.restype = ctypes.c_int
    lib.dcp_kv_cache_write.argtypes = [V, I64, V, V, I32, I32, I32, V, I64, I32, I32, V, I32, I32,
                                       I32, V, V]
    lib.dcp_topk_local.restype = ctypes.c_int
    lib.dcp_topk_local.argtypes = [V, I64, I32, V, I32, I32, I32, I32, V, V, V]
    lib.dcp_topk_merge.restype = ctypes.c_int
    lib.dcp_topk_merge.argtypes = [V, V, I32, I64, I32, I32, V, V, V]
    lib.mla_prefill_chunk_workspace_size.restype = SZ
    lib.mla_prefill_chunk_workspace_size.argtypes = [ctypes.POINTER(DecodeArgs), I32, I32]
    lib.mla_prefill_chunk_dcp.restype = ctypes.c_int
    lib.mla_prefill_chunk_dcp.argtypes = [ctypes.POINTER(DecodeArgs), I32, I32, V]
    lib.mla_decode_workspace_size.restype = SZ
    lib.mla_decode_workspace_size.argtypes = [ctypes.POINTER(DecodeArgs), I32, I32]
    if lib.dcp_abi_version() != DCP_ABI_VERSION:
        raise RuntimeError("libdcpmla ABI version mismatch")
    _lib = lib
    return lib


def _status_string(status: int) -> str:
    try:
        return load().dcp_status_string(int(status)).decode()
    except Exception:  # pragma: no cover
        return "status %d" % status


def _check(status: int, what: str):
    if status != DCP_OK:
        raise DcpError(status, what)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream, device=None) -> ctypes.c_void_p:
    """The stream handle a call runs on: `stream` (a torch.cuda.Stream or a raw handle), else
    the current stream of `device` (the device of the call's tensors)."""
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _i32(t: torch.Tensor, name: str):
    if t.dtype != torch.int32:
        raise ValueError("%s must be int32" % name)
    return t


# ------------------------------------------------------------------------------ remap
def dcp_remap_topk(global_idx: torch.Tensor, dcp: int, interleave: int, shard: int = -1,
                   local_idx: Optional[torch.Tensor] = None, count: Optional[torch.Tensor] = None,
                   stream=None):
    """Per-shard remap of global top-k slots -> (local_idx [n_out,R,K], count [n_out,R])."""
    _i32(global_idx, "global_idx")
    rows, k = global_idx.shape
    n_out = dcp if shard < 0 else 1
    if local_idx is None:
        local_idx = torch.empty((n_out, rows, k), dtype=torch.int32, device=global_idx.device)
    if count is None:
        count = torch.empty((n_out, rows), dtype=torch.int32, device=global_idx.device)
    _check(load().dcp_remap_topk(_ptr(global_idx), rows, k, dcp, interleave, shard,
                                 _ptr(local_idx), _ptr(count), _stream(stream, global_idx.device)),
           "dcp_remap_topk")
    return local_idx, count


def dcp_local_lengths(global_len: torch.Tensor, dcp: int, interleave: int, shard: int = -1,
                      local_len: Optional[torch.Tensor] = None, stream=None):
    """Local KV length per row on each shard (dense decode) -> [n_out, R] int32."""
    _i32(global_len, "global_len")
    rows = global_len.numel()
    n_out = dcp if shard < 0 else 1
    if local_len is None:
        local_len = torch.empty((n_out, rows), dtype=torch.int32, device=global_len.device)
    _check(load().dcp_local_lengths(_ptr(global_len), rows, dcp, interleave, shard,
                                    _ptr(local_len), _stream(stream, global_len.device)),
           "dcp_local_lengths")
    return local_len


# ------------------------------------------------------------------------------ DSA top-k producer
def dcp_topk_local(scores: torch.Tensor, local_len: torch.Tensor, k: int, dcp: int, interleave: int,
                   shard: int = -1, cand_score: Optional[torch.Tensor] = None,
                   cand_idx: Optional[torch.Tensor] = None, stream=None):
    """Each shard's best k local slots as global ids ascending with their scores:
    scores [n_in, R, stride] fp32, local_len [n_in, R] int32 ->
    (cand_score [n_in, R, k] fp32, cand_idx [n_in, R, k] int32)."""
    if scores.dtype != torch.float32 or scores.dim() != 3:
        raise ValueError("scores must be [n_in, rows, stride] float32")
    _i32(local_len, "local_len")
    n_in, rows, stride = scores.shape
    if n_in != (dcp if shard < 0 else 1) or local_len.shape != (n_in, rows):
        raise ValueError("scores / local_len do not match dcp and shard")
    if cand_score is None:
        cand_score = torch.empty((n_in, rows, k), dtype=torch.float32, device=scores.device)
    if cand_idx is None:
        cand_idx = torch.empty((n_in, rows, k), dtype=torch.int32, device=scores.device)
    _check(load().dcp_topk_local(_ptr(scores), rows, stride, _ptr(local_len), k, dcp, interleave,
                                 shard, _ptr(cand_score), _ptr(cand_idx),
                                 _stream(stream, scores.device)),
           "dcp_topk_local")
    return cand_score, cand_idx


def dcp_topk_merge(cand_score: torch.Tensor, cand_idx: torch.Tensor, k: Optional[int] = None,
                   topk: Optional[torch.Tensor] = None, count: Optional[torch.Tensor] = None,
                   stream=None):
    """Global top-k of a row from the D shards' lists [D, R, k_in] ->
    (topk [R, k] int32 ascending then -1, count [R] int32)."""
    if cand_score.dtype != torch.float32 or cand_score.dim() != 3:
        raise ValueError("cand_score must be [dcp, rows, k_in] float32")
    _i32(cand_idx, "cand_idx")
    D, rows, k_in = cand_score.shape
    if cand_idx.shape != cand_score.shape:
        raise ValueError("cand_idx must match cand_score")
    k = k_in if k is None else k
    if topk is None:
        topk = torch.empty((rows, k), dtype=torch.int32, device=cand_score.device)
    if count is None:
        count = torch.empty((rows,), dtype=torch.int32, device=cand_score.device)
    _check(load().dcp_topk_merge(_ptr(cand_score), _ptr(cand_idx), D, rows, k_in, k, _ptr(topk),
                                 _ptr(count), _stream(stream, cand_score.device)),
           "dcp_topk_merge")
    return topk, count


def dcp_topk_gather(cand_score: torch.Tensor, cand_idx: torch.Tensor, group=None):
    """The exchange step of the top-k producer on several ranks: rank s holds shard s's lists
    [1, R, k] (or [R, k]); returns every shard's lists [D, R, k] in shard (= rank) order,
    the input layout of dcp_topk_merge.  One all-gather per tensor of the process group."""
    import torch.distributed as dist
    D = dist.get_world_size(group)
    cs = cand_score.reshape(cand_score.shape[-2:]).contiguous()
    ci = cand_idx.reshape(cand_idx.shape[-2:]).contiguous()
    out_s = torch.empty((D,) + tuple(cs.shape), dtype=cs.dtype, device=cs.device)
    out_i = torch.empty((D,) + tuple(ci.shape), dtype=ci.dtype, device=ci.device)
    dist.all_gather(list(out_s.unbind(0)), cs, group=group)
    dist.all_gather(list(out_i.unbind(0)), ci, group=group)
    return out_s, out_i


# ------------------------------------------------------------------------------ cache write
def dcp_kv_cache_write(kv: torch.Tensor, seq: torch.Tensor, pos: torch.Tensor, kv_pool: torch.Tensor,
                       kv_dtype: int, block_table: torch.Tensor, dcp: int, interleave: int,
                       shard: int = -1, checked: bool = False, err_flag: Optional[torch.Tensor] = None,
                       stream=None):
    """Write token rows kv [n, 576] bf16 at (seq, pos) into kv_pool [pages, 64, bytes] (in
    place) on their owner shard; FP8 pools are quantised per 128 latent values."""
    if kv.dtype != torch.bfloat16 or kv.dim() != 2 or kv.shape[1] != 576:
        raise ValueError("kv must be [n, 576] bf16")
    _i32(seq, "seq")
    _i32(pos, "pos")
    _i32(block_table, "block_table")
    n = kv.shape[0]
    if seq.numel() != n or pos.numel() != n:
        raise ValueError("seq and pos must have n entries")
    num_pages, page_size = kv_pool.shape[0], kv_pool.shape[1]
    _check(load().dcp_kv_cache_write(_ptr(kv), n, _ptr(seq), _ptr(pos), dcp, interleave, shard,
                                     _ptr(kv_pool), num_pages, kv_dtype, page_size, _ptr(block_table),
                                     block_table.shape[1], block_table.shape[2], 1 if checked else 0,
                                     _ptr(err_flag), _stream(stream, kv.device)),
           "dcp_kv_cache_write")
    return kv_pool


# ------------------------------------------------------------------------------ merge
def dcp_lse_merge(part_out: torch.Tensor, part_lse: torch.Tensor, out: Optional[torch.Tensor] = None,
                  lse: Optional[torch.Tensor] = None, stream=None):
    """LSE merge of shard partials: [D,R,H,dv] fp32 + [D,R,H] -> ([R,H,dv] bf16, [R,H] fp32)."""
    D, R, H, dv = part_out.shape
    if part_out.dtype != torch.float32 or part_lse.dtype != torch.float32:
        raise ValueError("partials must be float32")
    if out is None:
        out = torch.empty((R, H, dv), dtype=torch.bfloat16, device=part_out.device)
    if lse is None:
        lse = torch.empty((R, H), dtype=torch.float32, device=part_out.device)
    _check(load().dcp_lse_merge(_ptr(part_out), _ptr(part_lse), D, R, H, dv, _ptr(out), _ptr(lse),
                                _stream(stream, part_out.device)), "dcp_lse_merge")
    return out, lse


# ------------------------------------------------------------------------------ decode
_ws_cache = {}


def _workspace(nbytes: int, device, stream: ctypes.c_void_p) -> Optional[torch.Tensor]:
    """A workspace reused by the calls on one (device, stream): calls on one stream run one
    after another, so they may share it; calls on different streams get their own."""
    if nbytes == 0:
        return None
    key = (str(device), stream.value)
    ws = _ws_cache.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.zeros(nbytes + 256, dtype=torch.uint8, device=device)
        _ws_cache[key] = ws
    return ws


def _decode_args(q, kv_pool, kv_dtype, block_table, row_seq, sm_scale, idx, count, kv_len,
                 max_kv_len, out, lse, num_splits, checked, err_flag, kernel_path=DCP_PATH_AUTO):
    if q.dtype != torch.bfloat16 or q.dim() != 3 or q.shape[2] != 576:
        raise ValueError("q must be [rows, heads, 576] bf16")
    if kv_pool.dtype != torch.uint8 or kv_pool.dim() != 3:
        raise ValueError("kv_pool must be [pages, page_size, token_bytes] uint8")
    if kv_pool.shape[2] != TOKEN_BYTES[kv_dtype]:
        raise ValueError("kv_pool token bytes do not match kv_dtype")
    _i32(block_table, "block_table")
    _i32(row_seq, "row_seq")
    a = DecodeArgs()
    a.q = _ptr(q).value
    a.rows = q.shape[0]
    a.heads = q.shape[1]
    a.sm_scale = float(sm_scale)
    a.kv_pool = _ptr(kv_pool).value
    a.num_pages = kv_pool.shape[0]
    a.kv_dtype = int(kv_dtype)
    a.page_size = kv_pool.shape[1]
    a.block_table = _ptr(block_table).value
    a.num_seqs = block_table.shape[-2]
    a.bt_stride = block_table.shape[-1]
    a.row_seq = _ptr(row_seq).value
    if idx is not None:
        _i32(idx, "idx")
        a.idx = _ptr(idx).value
        a.k = idx.shape[-1]
        if count is not None:
            a.count = _ptr(_i32(count, "count")).value
    elif kv_len is not None:
        if max_kv_len is None:
            raise ValueError("dense calls must pass max_kv_len, an upper bound of kv_len "
                             "(reading it from the device tensor would synchronise)")
        a.kv_len = _ptr(_i32(kv_len, "kv_len")).value
        a.max_kv_len = int(max_kv_len)
    a.out = _ptr(out).value
    a.lse = _ptr(lse).value
    a.num_splits = int(num_splits)
    a.checked = 1 if checked else 0
    a.err_flag = _ptr(err_flag).value if err_flag is not None else None
    a.kernel_path = int(kernel_path)
    return a


def mla_decode_workspace_size(args: DecodeArgs, num_shards_or_dcp: int, fused: bool) -> int:
    n = load().mla_decode_workspace_size(ctypes.byref(args), num_shards_or_dcp, 1 if fused else 0)
    if n == ctypes.c_size_t(-1).value:
        raise DcpError(DCP_ERR_INVALID_ARG, "mla_decode_workspace_size")
    return int(n)


def _bind_ws(a: DecodeArgs, n: int, fused: bool, device, workspace, stream):
    need = mla_decode_workspace_size(a, n, fused)
    if need:
        ws = workspace if workspace is not None else _workspace(need, device, stream)
        a.workspace = _ptr(ws).value
        a.workspace_bytes = ws.numel() * ws.element_size()
    return need


def mla_decode_partial_lse(q, kv_pool, kv_dtype, block_table, row_seq, sm_scale, *, idx=None,
                           count=None, kv_len=None, max_kv_len=None, num_shards=1, out=None,
                           lse=None, workspace=None, num_splits=0, checked=False, err_flag=None,
                           kernel_path=DCP_PATH_AUTO, stream=None):
    """Per-shard MLA decode with LSE.  block_table [S,B,maxp]; sparse: idx [S,R,K] local ids +
    count [S,R]; dense: kv_len [S,R] local lengths and max_kv_len >= all of them.
    Returns (out [S,R,H,512] fp32, lse [S,R,H])."""
    R, H, _ = q.shape
    if out is None:
        out = torch.empty((num_shards, R, H, 512), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((num_shards, R, H), dtype=torch.float32, device=q.device)
    a = _decode_args(q, kv_pool, kv_dtype, block_table, row_seq, sm_scale, idx, count, kv_len,
                     max_kv_len, out, lse, num_splits, checked, err_flag, kernel_path)
    st = _stream(stream, q.device)
    _bind_ws(a, num_shards, False, q.device, workspace, st)
    _check(load().mla_decode_partial_lse(ctypes.byref(a), num_shards, st), "mla_decode_partial_lse")
    return out, lse


def mla_decode_dcp_fused(q, kv_pool, kv_dtype, block_table, row_seq, sm_scale, dcp, interleave, *,
                         idx=None, kv_len=None, max_kv_len=None, out=None, lse=None,
                         workspace=None, num_splits=0, checked=False, err_flag=None,
                         kernel_path=DCP_PATH_AUTO, stream=None):
    """All shards of every row in one launch.  block_table [D,B,maxp]; sparse: idx [R,K] global
    slots (-1 pad); dense: kv_len [R] global lengths and max_kv_len >= all of them.
    Returns (out [R,H,512] bf16, lse [R,H])."""
    R, H, _ = q.shape
    if out is None:
        out = torch.empty((R, H, 512), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((R, H), dtype=torch.float32, device=q.device)
    a = _decode_args(q, kv_pool, kv_dtype, block_table, row_seq, sm_scale, idx, None, kv_len,
                     max_kv_len, out, lse, num_splits, checked, err_flag, kernel_path)
    st = _stream(stream, q.device)
    _bind_ws(a, dcp, True, q.device, workspace, st)
    _check(load().mla_decode_dcp_fused(ctypes.byref(a), dcp, interleave, st), "mla_decode_dcp_fused")
    return out, lse


def mla_prefill_chunk_dcp(q, kv_pool, kv_dtype, block_table, row_seq, sm_scale, dcp, interleave, *,
                          prefix_len, chunk_idx, max_prefix_len, out=None, lse=None, workspace=None,
                          stream=None):
    """Attention of a prefill chunk's query rows under DCP (the C entry of the same name):
    row r over its sequence's cached prefix [0, prefix_len[r]) and over the chunk slots
    chunk_idx[r] (global ids, -1 padded), per-shard partials merged by LSE.
    max_prefix_len bounds prefix_len on the host.  Returns (out [R, H, 512] bf16, lse [R, H])."""
    R, H, _ = q.shape
    if out is None:
        out = torch.empty((R, H, 512), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((R, H), dtype=torch.float32, device=q.device)
    a = _decode_args(q, kv_pool, kv_dtype, block_table, row_seq, sm_scale, chunk_idx, None, None,
                     None, out, lse, 0, False, None)
    a.kv_len = _ptr(_i32(prefix_len, "prefix_len")).value
    a.max_kv_len = int(max_prefix_len)
    need = load().mla_prefill_chunk_workspace_size(ctypes.byref(a), dcp, interleave)
    if need == ctypes.c_size_t(-1).value:
        raise DcpError(DCP_ERR_INVALID_ARG, "mla_prefill_chunk_workspace_size")
    st = _stream(stream, q.device)
    ws = workspace if workspace is not None else _workspace(need, q.device, st)
    a.workspace = _ptr(ws).value
    a.workspace_bytes = ws.numel() * ws.element_size()
    _check(load().mla_prefill_chunk_dcp(ctypes.byref(a), dcp, interleave, st), "mla_prefill_chunk_dcp")
    return out, lse


def mla_decode_dcp_fused_noalloc(q, kv_pool, kv_dtype, block_table, row_seq, sm_scale, dcp,
                                 interleave, *, out, lse, idx=None, kv_len=None, max_kv_len=None,
                                 num_splits=0, checked=False, err_flag=None, stream=None):
    """mla_decode_dcp_fused for callers that cannot allocate device memory.

    The caller passes preallocated outputs (out [R,H,512] bf16, lse [R,H] fp32); neither this
    function nor the library allocates anything: the split-KV scratch is a fixed
    DCP_NOALLOC_SCRATCH_BYTES array inside the library, shared by every call on a device.
    The first call on a device looks the array up, so make it before any stream capture;
    calls that overlap on the GPU race on the array.  A call that would need more scratch
    raises DcpError(DCP_ERR_WORKSPACE)."""
    if max_kv_len is None and kv_len is not None:
        raise ValueError("dense calls must pass max_kv_len (reading it from kv_len would sync)")
    a = _decode_args(q, kv_pool, kv_dtype, block_table, row_seq, sm_scale, idx, None, kv_len,
                     max_kv_len, out, lse, num_splits, checked, err_flag)
    _check(load().mla_decode_dcp_fused_noalloc(ctypes.byref(a), dcp, interleave,
                                               _stream(stream, q.device)),
           "mla_decode_dcp_fused_noalloc (static scratch %d bytes)" % DCP_NOALLOC_SCRATCH_BYTES)
    return out, lse
