"""Seeded synthetic inputs for the DCP MLA decode path.

This module is shared by the tests, the bench and the CPU oracle's callers.  It only
*draws* data: random queries, a paged latent KV pool, per-shard block tables, top-k
slot sets and merge partials.  It holds none of the path's arithmetic (no owner rule,
no slot remap, no attention, no merge); the single derived quantity it computes is a
generous *upper bound* on how many pages one shard may need for one sequence, which
only sizes the block tables.

Workloads follow the five decode configurations of the subject (dense/sparse MLA
decode with decode context parallelism):
  * Q, KV ~ N(0,1) cast to BF16;
  * FP8 KV: the 512 latent dims are stored as E4M3 with one fp32 scale per 128
    elements (scale = amax/448), the 64 RoPE dims stay BF16;
  * pages of 64 tokens; physical pages are a random permutation of the pool unless a
    contiguous layout is asked for;
  * top-k sets are distinct slots drawn uniformly from the row's visible range,
    padded with -1 when the range is shorter than k.

KV pool byte layout (one token row; a page is 64 consecutive token rows):
  BF16: 576 x bf16                       = 1152 B  (latent 0..511, RoPE 512..575)
  FP8 : 512 x e4m3 | 4 x fp32 | 64 x bf16 =  656 B  (latent, per-128 scales, RoPE)
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

KV_BF16 = 0
KV_FP8 = 1
PAGE_SIZE = 64
D_QK = 576          # 512 latent + 64 RoPE
D_V = 512           # values are the first 512 dims of the latent row
D_ROPE = 64
TOKEN_BYTES = {KV_BF16: 1152, KV_FP8: 656}
E4M3_MAX = 448.0
SM_SCALE = 1.0 / math.sqrt(192.0)


@dataclass
class DecodeProblem:
    """One batch of decode rows over a DCP-sharded paged KV pool (all tensors on one device)."""
    name: str
    rows: int
    heads: int
    dcp: int
    interleave: int           # 1 = token-interleaved owner, page_size = page-interleaved
    page_size: int
    kv_dtype: int
    sm_scale: float
    q: torch.Tensor           # [R, H, 576] bf16
    pool: torch.Tensor        # [num_pages, page_size, token_bytes] uint8
    block_table: torch.Tensor  # [D, B, max_pages] int32, -1 = unused
    row_seq: torch.Tensor     # [R] int32: sequence (block-table row) of each decode row
    row_len: torch.Tensor     # [R] int32: visible global length of each decode row
    topk: Optional[torch.Tensor]  # [R, K] int32 global slots (-1 padded) or None (dense)
    seq_len: torch.Tensor     # [B] int32
    meta: dict = field(default_factory=dict)

    @property
    def k(self) -> int:
        return 0 if self.topk is None else int(self.topk.shape[1])

    @property
    def num_seqs(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def token_bytes(self) -> int:
        return TOKEN_BYTES[self.kv_dtype]

    def to(self, device) -> "DecodeProblem":
        def mv(t):
            return None if t is None else t.to(device)
        return DecodeProblem(self.name, self.rows, self.heads, self.dcp, self.interleave,
                             self.page_size, self.kv_dtype, self.sm_scale, mv(self.q),
                             mv(self.pool), mv(self.block_table), mv(self.row_seq),
                             mv(self.row_len), mv(self.topk), mv(self.seq_len), dict(self.meta))


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def pages_bound(seq_len: int, dcp: int, interleave: int, page_size: int) -> int:
    """Upper bound on the pages any one shard needs for a sequence of seq_len tokens.

    A shard never holds more than interleave * ceil(seq_len / (interleave * dcp)) tokens
    of a sequence under either interleave rule; one spare page is added.
    """
    per_shard = interleave * -(-seq_len // (interleave * dcp))
    return -(-per_shard // page_size) + 1


def make_block_tables(seq_lens, dcp, interleave, page_size, gen, device, permute=True):
    """Per-shard block tables over one shared physical page pool.

    Returns (block_table [D, B, maxp] int32 with -1 for unused entries, num_pages).
    Every (shard, sequence) gets pages_bound(...) distinct physical pages.
    """
    need = [pages_bound(int(L), dcp, interleave, page_size) for L in seq_lens]
    maxp = max(need)
    B = len(seq_lens)
    total = dcp * sum(need)
    if permute:
        phys = torch.randperm(total, generator=gen, device=gen.device).to(torch.int32)
    else:
        phys = torch.arange(total, dtype=torch.int32, device=gen.device)
    bt = torch.full((dcp, B, maxp), -1, dtype=torch.int32, device=gen.device)
    cur = 0
    for s in range(dcp):
        for b in range(B):
            n = need[b]
            bt[s, b, :n] = phys[cur:cur + n]
            cur += n
    return bt.to(device), total


def fill_pool(num_pages, page_size, kv_dtype, gen, chunk_tokens=1 << 20):
    """A pool of num_pages pages whose every token row is N(0,1) data in the pool format."""
    dev = gen.device
    n_tok = num_pages * page_size
    tb = TOKEN_BYTES[kv_dtype]
    pool = torch.empty((n_tok, tb), dtype=torch.uint8, device=dev)
    for start in range(0, n_tok, chunk_tokens):
        n = min(chunk_tokens, n_tok - start)
        if kv_dtype == KV_BF16:
            x = torch.randn((n, D_QK), generator=gen, device=dev, dtype=torch.float32)
            pool[start:start + n] = x.to(torch.bfloat16).view(torch.uint8).view(n, tb)
        else:
            lat = torch.randn((n, D_V), generator=gen, device=dev, dtype=torch.float32)
            rope = torch.randn((n, D_ROPE), generator=gen, device=dev, dtype=torch.float32)
            codes, scales = quantize_e4m3_per128(lat)
            pool[start:start + n, 0:512] = codes.view(torch.uint8)
            pool[start:start + n, 512:528] = scales.contiguous().view(torch.uint8).view(n, 16)
            pool[start:start + n, 528:656] = rope.to(torch.bfloat16).view(torch.uint8).view(n, 128)
            del lat, rope, codes, scales
    return pool.view(num_pages, page_size, tb)


def quantize_e4m3_per128(lat: torch.Tensor):
    """Store fp32 latent rows [n, 512] as E4M3 codes with one fp32 scale per 128 values.

    scale = amax / 448 per block (a block of zeros gets scale 0 and zero codes); the
    codes are round-to-nearest-even of x / scale, clamped to +-448.  This is the
    cache-writer's job in a serving system; here it only produces test data.
    """
    n = lat.shape[0]
    blk = lat.view(n, 4, 128)
    amax = blk.abs().amax(dim=-1)
    scale = amax / E4M3_MAX
    safe = torch.where(scale > 0, scale, torch.ones_like(scale))
    y = (blk / safe.unsqueeze(-1)).clamp(-E4M3_MAX, E4M3_MAX)
    y = torch.where(scale.unsqueeze(-1) > 0, y, torch.zeros_like(y))
    codes = y.to(torch.float8_e4m3fn).view(n, 512)
    return codes, scale.to(torch.float32)


def sample_topk(row_len: torch.Tensor, k: int, gen, sort=False):
    """k distinct slots per row drawn uniformly from [0, row_len); -1 pads short rows."""
    dev = gen.device
    R = row_len.numel()
    maxlen = int(row_len.max().item())
    keys = torch.rand((R, maxlen), generator=gen, device=dev)
    pos = torch.arange(maxlen, device=dev).unsqueeze(0)
    keys = torch.where(pos < row_len.to(dev).unsqueeze(1), keys, torch.full_like(keys, 2.0))
    kk = min(k, maxlen)
    vals, idx = torch.topk(keys, kk, dim=1, largest=False, sorted=True)
    idx = torch.where(vals < 1.5, idx, torch.full_like(idx, -1)).to(torch.int32)
    if kk < k:
        idx = torch.cat([idx, torch.full((R, k - kk), -1, dtype=torch.int32, device=dev)], 1)
    if sort:
        big = torch.where(idx < 0, torch.full_like(idx, 2**31 - 1), idx)
        big, _ = torch.sort(big, dim=1)
        idx = torch.where(big == 2**31 - 1, torch.full_like(big, -1), big)
    return idx.contiguous()


def make_decode_problem(name, seq_lens, heads, k, kv_dtype, dcp, interleave=1,
                        mtp=1, seed=0, device="cpu", permute_pages=True,
                        page_size=PAGE_SIZE, sm_scale=SM_SCALE, sort_topk=False):
    """Build a DecodeProblem.

    seq_lens: per-sequence context length.  mtp: query tokens per sequence; token i of a
    sequence of length L sees L - (mtp - 1) + i tokens (MTP-style causal visibility).
    k: top-k size for sparse attention, or None for dense attention over the visible range.
    Data are drawn on `device` (generation on a GPU is much faster at full size).
    """
    gen = _gen(seed, device)
    seq_lens = [int(x) for x in seq_lens]
    B = len(seq_lens)
    bt, num_pages = make_block_tables(seq_lens, dcp, interleave, page_size, gen, device,
                                      permute=permute_pages)
    pool = fill_pool(num_pages, page_size, kv_dtype, gen)
    R = B * mtp
    row_seq = torch.arange(B, dtype=torch.int32, device=device).repeat_interleave(mtp)
    row_len = torch.tensor([L - (mtp - 1) + i for L in seq_lens for i in range(mtp)],
                           dtype=torch.int32, device=device)
    q = torch.randn((R, heads, D_QK), generator=gen, device=device).to(torch.bfloat16)
    topk = None if k is None else sample_topk(row_len, k, gen, sort=sort_topk)
    return DecodeProblem(name, R, heads, dcp, interleave, page_size, kv_dtype, float(sm_scale),
                         q, pool, bt, row_seq, row_len, topk,
                         torch.tensor(seq_lens, dtype=torch.int32, device=device),
                         {"seed": seed, "mtp": mtp})


# ---------------------------------------------------------------------------------------
# The five workloads (full size) and scaled-down parity variants.
# ---------------------------------------------------------------------------------------

def cfg1_tiny_dense(device="cpu"):
    """Tiny dense MLA decode, BF16: 2 rows, 16 heads, 256 tokens, contiguous pages, D=2."""
    return make_decode_problem("cfg1_tiny_dense_bf16", [256, 256], 16, None, KV_BF16, 2, 1,
                               seed=0, device=device, permute_pages=False)


def _uniform_lens(n, lo, hi, seed):
    g = torch.Generator().manual_seed(seed + 1000)
    return torch.randint(lo, hi + 1, (n,), generator=g).tolist()


def cfg2_sparse_topk512(device="cpu"):
    """Sparse top-k 512, BF16 KV: 16 rows, 64 heads, lengths U[8192, 32768], D=4."""
    return make_decode_problem("cfg2_sparse_topk512_bf16", _uniform_lens(16, 8192, 32768, 1),
                               64, 512, KV_BF16, 4, 1, seed=1, device=device)


def cfg3_sparse_topk2048_fp8(device="cpu", seqs=64, seq_len=131072):
    """Sparse top-k 2048, FP8 KV: 64 seqs x 6 MTP rows, 128 heads, 131072 tokens, D=8."""
    return make_decode_problem("cfg3_sparse_topk2048_fp8", [seq_len] * seqs, 128, 2048, KV_FP8,
                               8, 1, mtp=6, seed=2, device=device)


def cfg5_dense_long(device="cpu", seqs=32, lo=16384, hi=65536):
    """Long-context dense MLA decode, BF16 KV: 32 rows, 128 heads, U[16384, 65536], D=4."""
    return make_decode_problem("cfg5_dense_long_bf16", _uniform_lens(seqs, lo, hi, 4), 128, None,
                               KV_BF16, 4, 1, seed=4, device=device)


@dataclass
class RemapMergeProblem:
    """Remap + merge stress inputs (no KV)."""
    dcp: int
    interleave: int
    topk: torch.Tensor        # [R, K] int32, ascending valid ids then -1 padding
    part_out: torch.Tensor    # [D, R, H, 512] fp32
    part_lse: torch.Tensor    # [D, R, H] fp32 (-inf marks an empty shard)


def cfg4_remap_merge(dcp, device="cpu", rows=256, k=2048, heads=128, seq_len=131072,
                     interleave=PAGE_SIZE, seed=3, with_partials=True):
    """Remap + merge stress: 256 rows x 2048 sorted global ids, ~10% -1 padded rows,
    ~5% rows whose ids all lie below (dcp-1)*interleave, one all-padding row;
    partials N(0,1) fp32 with LSE ~ N(5,3) and ~5% (shard,row) pairs empty (-inf)."""
    gen = _gen(seed + 17 * dcp, device)
    row_len = torch.full((rows,), seq_len, dtype=torch.int32, device=device)
    topk = sample_topk(row_len, k, gen, sort=True)
    u = torch.rand((rows,), generator=gen, device=device)
    # ~10% of rows keep a U[1, k) prefix of valid ids
    nvalid = torch.randint(1, k, (rows,), generator=gen, device=device)
    pos = torch.arange(k, device=device).unsqueeze(0)
    pad_rows = u < 0.10
    topk = torch.where(pad_rows.unsqueeze(1) & (pos >= nvalid.unsqueeze(1)),
                       torch.full_like(topk, -1), topk)
    # ~5% of rows draw all ids below (dcp-1)*interleave
    low = (u >= 0.10) & (u < 0.15)
    span = max(1, (dcp - 1) * interleave)
    if dcp > 1 and bool(low.any()):
        nl = int(low.sum())
        lens = torch.full((nl,), span, dtype=torch.int32, device=device)
        topk[low] = sample_topk(lens, k, gen, sort=True)
    topk[rows // 2] = -1      # one row empty on every shard
    part_out = part_lse = None
    if with_partials:
        part_out = torch.randn((dcp, rows, heads, D_V), generator=gen, device=device)
        part_lse = 5.0 + 3.0 * torch.randn((dcp, rows, heads), generator=gen, device=device)
        empty = torch.rand((dcp, rows), generator=gen, device=device) < 0.05
        empty[:, rows // 2] = True
        part_lse = torch.where(empty.unsqueeze(-1), torch.full_like(part_lse, -math.inf), part_lse)
        part_out = torch.where(empty[..., None, None], torch.zeros_like(part_out), part_out)
    return RemapMergeProblem(dcp, interleave, topk.contiguous(), part_out, part_lse)


# ---------------------------------------------------------------------------------------
# DSA indexer scores for the top-k producer (per-shard candidate lists and their merge).
# ---------------------------------------------------------------------------------------

@dataclass
class TopkProducerProblem:
    """Indexer scores of every shard's local slots for a batch of decode rows."""
    dcp: int
    interleave: int
    k: int
    row_len: torch.Tensor     # [R] int32 visible global length of each row
    scores: torch.Tensor      # [D, R, stride] fp32, N(0,1); entries past a row's local length unused
    stride: int               # >= the longest local length (an upper bound, see local_len_bound)


def local_len_bound(seq_len: int, dcp: int, interleave: int) -> int:
    """Upper bound on the slots any one shard holds of seq_len global slots."""
    return interleave * -(-seq_len // (interleave * dcp))


def index_scores(shards: int, rows: int, stride: int, gen, ties: bool = False,
                 masked: float = 0.0) -> torch.Tensor:
    """Indexer scores N(0,1) fp32 [shards, rows, stride]; ties=True rounds them to
    multiples of 1/4 (many equal scores); a fraction `masked` is set to -inf."""
    s = torch.randn((shards, rows, stride), generator=gen, device=gen.device)
    if ties:
        s = torch.round(s * 4.0) / 4.0
    if masked > 0:
        s = torch.where(torch.rand(s.shape, generator=gen, device=gen.device) < masked,
                        torch.full_like(s, float("-inf")), s)
    return s.contiguous()


def topk_producer_topk2048(device="cpu", seqs=64, mtp=6, seq_len=131072, dcp=8, k=2048,
                           interleave=1, seed=6):
    """The top-k 2048 decode batch's producer: 64 sequences x 6 MTP rows (row i of a
    sequence sees seq_len - 5 + i slots), D = 8 shards, N(0,1) indexer scores."""
    gen = _gen(seed, device)
    row_len = torch.tensor([seq_len - (mtp - 1) + i for _ in range(seqs) for i in range(mtp)],
                           dtype=torch.int32, device=device)
    stride = local_len_bound(seq_len, dcp, interleave)
    scores = index_scores(dcp, seqs * mtp, stride, gen)
    return TopkProducerProblem(dcp, interleave, k, row_len, scores, stride)


# ---------------------------------------------------------------------------------------
# Chunked prefill: the query rows of one prefill chunk per sequence.
# ---------------------------------------------------------------------------------------

def prefill_chunk_problem(name, prefix_lens, chunk, heads, kv_dtype, dcp, interleave=1, seed=7,
                          device="cpu"):
    """Sequences of prefix_lens[b] cached tokens followed by a chunk of `chunk` new tokens
    (all already in the pool); one query row per chunk token, row i of a chunk seeing the
    prefix and chunk tokens 0..i (a dense problem whose row i sees prefix + i + 1 slots)."""
    return make_decode_problem(name, [int(p) + chunk for p in prefix_lens], heads, None, kv_dtype,
                               dcp, interleave, mtp=chunk, seed=seed, device=device)


def prefill_chunk_inputs(prob: DecodeProblem, chunk: int):
    """Per row of a prefill_chunk_problem: the cached-prefix length [R] int32 and the chunk
    slots the row sees [R, chunk] int32 (global ids prefix .. prefix + i, then -1)."""
    dev = prob.q.device
    L = prob.seq_len.to(dev)[prob.row_seq.long()]
    prefix = (L - chunk).to(torch.int32)
    i = torch.arange(prob.rows, device=dev) % chunk
    c = torch.arange(chunk, device=dev)
    ids = prefix.unsqueeze(1).to(torch.int64) + c.unsqueeze(0)
    ids = torch.where(c.unsqueeze(0) <= i.unsqueeze(1), ids, torch.full_like(ids, -1))
    return prefix.contiguous(), ids.to(torch.int32).contiguous()


def prefill_chunk_fp8(device="cpu", seqs=2, prefix=16384, chunk=64, heads=128, dcp=8):
    """A prefill chunk of the top-k 2048 decode model's shapes: 2 sequences x 64 chunk tokens
    after a 16384-token cached prefix, 128 heads, FP8 KV, D = 8 token-interleaved."""
    return prefill_chunk_problem("prefill_chunk_fp8", [prefix] * seqs, chunk, heads, KV_FP8, dcp,
                                 1, seed=7, device=device)
