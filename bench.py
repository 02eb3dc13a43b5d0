"""Benchmark of the DCP sparse MLA decode hot path on one GB300 (or N replicas).

A step is one fused decode launch (remap to owner shards, attention over every shard's
paged FP8 KV, on-chip LSE merge) over the batch of the top-k-2048 / 128-head / FP8 KV
workload: 64 sequences x 6 MTP query rows, 131072-token contexts, DCP = 8 token-
interleaved shards.  The unfused pipeline (remap -> per-shard partials -> merge) is timed
beside it.  Inputs are resident in HBM; L2 is flushed (256 MB write) between steps and
each step is timed alone with CUDA events on the launching stream.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line.  --impl reference times the CPU oracle on a bounded sample of the
same workload instead.
"""
import argparse
import json
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "sparse MLA decode rows/s + achieved HBM TB/s, top-k 2048, 128 heads, FP8 KV"
WORKLOAD = "sparse MLA decode top-k 2048, 128 heads, FP8 E4M3 KV (per-128 scales), " \
           "64 seqs x 6 MTP rows = 384 rows, context 131072, page 64, DCP=8 token-interleaved"
BYTES_PER_SLOT = 656          # FP8 KV row gathered once per (row, selected slot)
D_QK, D_V = 576, 512


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "src": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "src": "fallback"}


class ClockSampler:
    """SM clock and clock-event (throttle) reasons sampled every ~2 ms through NVML (read-only
    queries via ctypes) in a background thread while the timed region runs.  Without NVML it
    records no samples and says so in its result."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, dev):
        import ctypes
        self.dev = dev
        self.samples = []
        self.reasons = set()
        self.max_mhz = None
        self._stop = threading.Event()
        self.nvml = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            h = ctypes.c_void_p()
            props = torch.cuda.get_device_properties(dev)
            ok = False
            if hasattr(props, "pci_bus_id"):
                bus = ("%08X:%02X:%02X.0" % (getattr(props, "pci_domain_id", 0), props.pci_bus_id,
                                              getattr(props, "pci_device_id", 0))).encode()
                ok = nv.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(h)) == 0
            if not ok and nv.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(h)) != 0:
                raise OSError("no NVML handle")
            self.nvml, self.h, self.ct = nv, h, ctypes
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            self._reasons_fn = fn
        except Exception:
            self.nvml = None

    def _run(self):
        ct, nv, h = self.ct, self.nvml, self.h
        mhz = ct.c_uint()
        rs = ct.c_ulonglong()
        while not self._stop.is_set():
            if nv.nvmlDeviceGetClockInfo(h, 1, ct.byref(mhz)) == 0:
                self.samples.append(float(mhz.value))
            if self._reasons_fn(h, ct.byref(rs)) == 0:
                for bit, name in self.REASONS.items():
                    if rs.value & bit:
                        self.reasons.add(name)
            time.sleep(0.002)

    def start(self):
        if self.nvml is not None:
            self.t = threading.Thread(target=self._run, daemon=True)
            self.t.start()

    def stop(self):
        if self.nvml is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["NVML unavailable"],
                    "samples": 0}
        self._stop.set()
        self.t.join()
        busy = self.samples
        return {"sm_mhz": statistics.median(busy) if busy else None, "sm_max_mhz": self.max_mhz,
                "reasons": sorted(self.reasons), "samples": len(busy), "source": "nvml"}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# DRAM traffic of the decode kernel (dram__bytes_read.sum + dram__bytes_write.sum) from one ncu
# capture of a 96-row slice of this workload (bench.py --seqs 16), per decode row; the bench
# scales it to the full launch by rows, since the traffic grows with the rows processed.
TRAFFIC_CAPTURE = {"bytes_per_row": (168.456448e6 + 18.000896e6) / 96, "rows": 96,
                   "kernel": "decode_tc_kernel<FP8, fused, sparse>"}


def make_workload(dev, seqs=64):
    import synth
    return synth.cfg3_sparse_topk2048_fp8(device=dev, seqs=seqs)


def algorithmic(prob):
    valid = int((prob.topk >= 0).sum().item())
    return valid * BYTES_PER_SLOT, valid * 2.0 * prob.heads * (D_QK + D_V), valid


def host_copy(prob):
    """The same workload with every tensor in host memory (for the CPU oracle)."""
    return prob.to("cpu")


def time_oracle_rows(prob_host, seconds):
    """Oracle on as many rows of the workload as fit in about `seconds` of host time."""
    import oracle
    oracle.build()
    t0 = time.perf_counter()
    oracle.attention_problem(prob_host, rows=[0])
    t1 = time.perf_counter() - t0
    return max(1, min(prob_host.rows, int(seconds / max(t1, 1e-4))))


def run_reference(args):
    """The CPU oracle, as it stands, on a bounded sample of the same workload per step."""
    import oracle
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    prob = host_copy(make_workload(dev))
    per_step = min(8.0, 150.0 / max(1, args.steps + args.warmup))
    n = time_oracle_rows(prob, per_step)
    rows = list(range(n))
    for _ in range(args.warmup):
        oracle.attention_problem(prob, rows=rows)
    times = []
    for _ in range(args.steps):
        t = time.perf_counter()
        oracle.attention_problem(prob, rows=rows)
        times.append(time.perf_counter() - t)
    total = sum(times)
    val = n * len(times) / total
    cores = oracle.num_threads()
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "rows/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "rows_per_step": n, "parallelism": "cpu oracle"},
            "cpu_baseline": {"value": val, "unit": "rows/s", "cores": cores, "kind": "oracle",
                             "sample": "%d of the 384 decode rows per step" % n},
            "e2e": {"value": val, "unit": "rows/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def time_kv_cache_write(dcp, dev, peaks, stream, flush, steps):
    """The cache-fill call before the path: 64 sequences x 2048 new tokens written into an FP8
    pool (D = 8, token-interleaved), timed like the decode (events, L2 flushed between
    calls).  Algorithmic bytes per row: 1152 read + 8 (sequence, position) + 656 written."""
    seqs, T, D = 64, 2048, 8
    gen = torch.Generator(device=dev).manual_seed(7)
    pages = D * seqs * (T // D // 64)
    bt = torch.randperm(pages, device=dev, generator=gen).to(torch.int32).view(D, seqs, -1)
    kv = torch.randn((seqs * T, 576), device=dev, generator=gen).to(torch.bfloat16)
    seq = torch.arange(seqs, device=dev, dtype=torch.int32).repeat_interleave(T)
    pos = torch.arange(T, device=dev, dtype=torch.int32).repeat(seqs)
    pool = torch.zeros((pages, 64, 656), dtype=torch.uint8, device=dev)

    def call():
        dcp.dcp_kv_cache_write(kv, seq, pos, pool, 1, bt, D, 1)

    for _ in range(3):
        call()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(max(3, steps))]
    for a, b in evs:
        flush.fill_(3)
        a.record(stream)
        call()
        b.record(stream)
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    nbytes = seqs * T * (1152 + 8 + 656)
    gbs = nbytes / (ms / 1e3) / 1e9
    return {"rows": seqs * T, "kv_dtype": "fp8_e4m3_per128_scale", "dcp": D, "us": 1e3 * ms,
            "algorithmic_bytes": nbytes, "achieved_gbs": gbs, "peak_gbs": peaks["hbm_gbs"],
            "frac": gbs / peaks["hbm_gbs"], "bound": "hbm", "launches_per_call": 1}


def time_topk_producer(dcp, dev, peaks, stream, flush, steps, seqs=64):
    """The DSA top-k producer of the decode batch: every shard's candidate list (8 shards x
    384 rows, 16384 local slots each, k = 2048) and their merge into the rows' global top-k,
    timed like the decode (events, L2 flushed between calls).  Algorithmic bytes: the local
    scores read (4 B per local slot) and the lists written (8 B per candidate); the lists
    read again (8 B) and the top-k written (4 B per entry + 4 B count per row)."""
    import synth
    p = synth.topk_producer_topk2048(device=dev, seqs=seqs)
    D, k = p.dcp, p.k
    R = p.row_len.numel()
    ll = dcp.dcp_local_lengths(p.row_len, D, p.interleave)
    cs = torch.empty((D, R, k), dtype=torch.float32, device=dev)
    ci = torch.empty((D, R, k), dtype=torch.int32, device=dev)
    top = torch.empty((R, k), dtype=torch.int32, device=dev)
    cnt = torch.empty((R,), dtype=torch.int32, device=dev)

    def local():
        dcp.dcp_topk_local(p.scores, ll, k, D, p.interleave, cand_score=cs, cand_idx=ci)

    def merge():
        dcp.dcp_topk_merge(cs, ci, k, topk=top, count=cnt)

    for _ in range(3):
        local()
        merge()
    n = max(3, steps)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
    for a, b, c in ev:
        flush.fill_(4)
        a.record(stream)
        local()
        b.record(stream)
        merge()
        c.record(stream)
    torch.cuda.synchronize()
    ms_l = statistics.mean(a.elapsed_time(b) for a, b, _ in ev)
    ms_m = statistics.mean(b.elapsed_time(c) for _, b, c in ev)
    b_local = int(ll.sum().item()) * 4 + D * R * 4 + D * R * k * 8
    b_merge = D * R * k * 8 + R * k * 4 + R * 4
    g_l = b_local / (ms_l / 1e3) / 1e9
    g_m = b_merge / (ms_m / 1e3) / 1e9
    g = (b_local + b_merge) / ((ms_l + ms_m) / 1e3) / 1e9
    return {"workload": "DSA top-k producer, 8 shards x 384 rows x 16384 local slots, k 2048",
            "us_local": 1e3 * ms_l, "us_merge": 1e3 * ms_m,
            "algorithmic_bytes_local": b_local, "algorithmic_bytes_merge": b_merge,
            "achieved_gbs_local": g_l, "achieved_gbs_merge": g_m, "achieved_gbs": g,
            "peak_gbs": peaks["hbm_gbs"], "frac": g / peaks["hbm_gbs"], "bound": "hbm",
            "launches_per_call": 2}


def _timed_us(stream, flush, fn, steps, fill):
    """Mean device time of fn in µs: fn is recorded once into a CUDA graph, which is replayed
    max(3, steps) times after 3 warm-up replays, each replay timed with CUDA events on the
    launching stream and preceded by an L2 flush (the graph keeps the binding's host-side
    work out of the timing of the small configurations)."""
    fn()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(stream.device)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            fn()
    stream.wait_stream(side)
    for _ in range(3):
        graph.replay()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(max(3, steps))]
    for a, b in ev:
        flush.fill_(fill)
        a.record(stream)
        graph.replay()
        b.record(stream)
    torch.cuda.synchronize()
    return 1e3 * statistics.mean(a.elapsed_time(b) for a, b in ev)


def time_configs(dcp, dev, peaks, stream, flush, steps):
    """Every synthetic configuration of the hot path at N = 1 besides the headline one: the
    decode configurations (tiny dense BF16, sparse top-k 512 BF16, long dense BF16) fused and
    unfused (remap or local lengths -> per-shard partials -> merge), with rows/s, µs per call
    (one layer) and the fraction of the roofline max(gathered KV bytes / HBM peak, FLOPs /
    tensor peak); and the remap + merge stress at D = 2, 4, 8 against HBM.  Inputs as the
    parity tests draw them; each call replayed from a CUDA graph, L2 flushed before it."""
    import synth
    res = {}
    for name, make in (("cfg1_tiny_dense_bf16", synth.cfg1_tiny_dense),
                       ("cfg2_sparse_topk512_bf16", synth.cfg2_sparse_topk512),
                       ("cfg5_dense_long_bf16", synth.cfg5_dense_long)):
        g = make(device=dev)
        R, H, D, I = g.rows, g.heads, g.dcp, g.interleave
        if g.topk is not None:
            slots = int((g.topk >= 0).sum().item())
            kw = dict(idx=g.topk)
        else:
            slots = int(g.row_len.sum().item())
            kw = dict(kv_len=g.row_len, max_kv_len=int(g.row_len.max().item()))
            ll = dcp.dcp_local_lengths(g.row_len, D, I)
        out = torch.empty((R, H, 512), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((R, H), dtype=torch.float32, device=dev)
        po = torch.empty((D, R, H, 512), dtype=torch.float32, device=dev)
        pl = torch.empty((D, R, H), dtype=torch.float32, device=dev)
        loc = torch.empty((D, R, max(g.k, 1)), dtype=torch.int32, device=dev)
        cnt = torch.empty((D, R), dtype=torch.int32, device=dev)

        def fused():
            dcp.mla_decode_dcp_fused(g.q, g.pool, g.kv_dtype, g.block_table, g.row_seq,
                                     g.sm_scale, D, I, out=out, lse=lse, **kw)

        def unfused():
            if g.topk is not None:
                dcp.dcp_remap_topk(g.topk, D, I, local_idx=loc, count=cnt)
                dcp.mla_decode_partial_lse(g.q, g.pool, g.kv_dtype, g.block_table, g.row_seq,
                                           g.sm_scale, idx=loc, count=cnt, num_shards=D,
                                           out=po, lse=pl)
            else:
                dcp.mla_decode_partial_lse(g.q, g.pool, g.kv_dtype, g.block_table, g.row_seq,
                                           g.sm_scale, kv_len=ll, max_kv_len=kw["max_kv_len"],
                                           num_shards=D, out=po, lse=pl)
            dcp.dcp_lse_merge(po, pl, out=out, lse=lse)

        us_f = _timed_us(stream, flush, fused, steps, 6)
        us_u = _timed_us(stream, flush, unfused, steps, 7)
        kv_bytes = slots * g.token_bytes
        flops = slots * 2 * H * (576 + 512)
        t_hbm = kv_bytes / (peaks["hbm_gbs"] * 1e9) * 1e6
        t_tc = flops / (peaks["bf16_tflops"] * 1e12) * 1e6
        roof = max(t_hbm, t_tc)
        res[name] = {"rows": R, "heads": H, "dcp": D, "kv_slots": slots,
                     "kernel": "tensor cores" if 48 <= H <= 128 else "CUDA cores",
                     "fused": {"us": us_f, "rows_per_s": R / (us_f / 1e6),
                               "roofline_frac": roof / us_f},
                     "unfused": {"us": us_u, "rows_per_s": R / (us_u / 1e6),
                                 "roofline_frac": roof / us_u},
                     "bound": "tensor" if t_tc >= t_hbm else "hbm", "roofline_us": roof,
                     "algorithmic_bytes": kv_bytes, "flops": flops}
        del g
    stress = {}
    for D in (2, 4, 8):
        m = synth.cfg4_remap_merge(D, device=dev)
        R, K = m.topk.shape
        H = m.part_out.shape[2]
        loc = torch.empty((D, R, K), dtype=torch.int32, device=dev)
        cnt = torch.empty((D, R), dtype=torch.int32, device=dev)
        out = torch.empty((R, H, 512), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((R, H), dtype=torch.float32, device=dev)
        us_r = _timed_us(stream, flush, lambda: dcp.dcp_remap_topk(
            m.topk, D, m.interleave, local_idx=loc, count=cnt), steps, 8)
        us_m = _timed_us(stream, flush, lambda: dcp.dcp_lse_merge(
            m.part_out, m.part_lse, out=out, lse=lse), steps, 9)
        b_r = R * K * 4 + D * R * K * 4 + D * R * 4
        b_m = D * R * H * (512 + 1) * 4 + R * H * (512 * 2 + 4)
        stress["dcp%d" % D] = {
            "remap_us": us_r, "remap_gbs": b_r / (us_r / 1e6) / 1e9,
            "merge_us": us_m, "merge_gbs": b_m / (us_m / 1e6) / 1e9,
            "merge_frac": b_m / (us_m / 1e6) / 1e9 / peaks["hbm_gbs"],
            "remap_bytes": b_r, "merge_bytes": b_m}
        del m
    res["cfg4_remap_merge_stress"] = dict(stress, rows=256, k=2048, heads=128,
                                          interleave="page (64)", bound="hbm")
    return res


def time_prefill_chunk(dcp, dev, peaks, stream, flush, steps):
    """A chunked-prefill step of the same model shapes: 2 sequences x 64 chunk tokens after a
    16384-token cached prefix, 128 heads, FP8, D = 8.  Timed as the prefix + chunk partials
    merged by LSE (the composition) and as one fused dense launch over the same lengths.
    FLOPs: 2*H*(576+512) per (row, visible slot)."""
    import synth
    prob = synth.prefill_chunk_fp8(device=dev)
    chunk = 64
    prefix, ids = synth.prefill_chunk_inputs(prob, chunk)
    pmax = int(prefix.max().item())
    lmax = int(prob.row_len.max().item())
    out = torch.empty((prob.rows, prob.heads, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((prob.rows, prob.heads), dtype=torch.float32, device=dev)

    def composed():
        dcp.mla_prefill_chunk_dcp(prob.q, prob.pool, prob.kv_dtype, prob.block_table, prob.row_seq,
                                  prob.sm_scale, prob.dcp, prob.interleave, prefix_len=prefix,
                                  chunk_idx=ids, max_prefix_len=pmax, out=out, lse=lse)

    def fused():
        dcp.mla_decode_dcp_fused(prob.q, prob.pool, prob.kv_dtype, prob.block_table, prob.row_seq,
                                 prob.sm_scale, prob.dcp, prob.interleave, kv_len=prob.row_len,
                                 max_kv_len=lmax, out=out, lse=lse)

    res = {}
    flops = 2.0 * prob.heads * (D_QK + D_V) * float(prob.row_len.sum().item())
    for name, f in (("composed", composed), ("fused_dense", fused)):
        for _ in range(3):
            f()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(max(3, steps // 2))]
        for a, b in evs:
            flush.fill_(5)
            a.record(stream)
            f()
            b.record(stream)
        torch.cuda.synchronize()
        ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
        tf = flops / (ms / 1e3) / 1e12
        res[name] = {"us": 1e3 * ms, "chunk_tokens_per_s": prob.rows / (ms / 1e3),
                     "tflops": tf, "frac": tf / peaks["bf16_tflops"]}
    res["workload"] = ("chunked prefill, 2 seqs x 64 chunk tokens after a 16384-token prefix, "
                       "128 heads, FP8, DCP=8")
    res["bound"] = "tensor"
    res["peak_tflops"] = peaks["bf16_tflops"]
    return res


def max_over_ranks(x: float, device) -> float:
    """The largest of every rank's x (x itself without a process group)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: int, steps: int, max_total_ms: float, world: int) -> float:
    """Units all ranks processed per second, over the slowest rank's time."""
    return world * units_per_rank * steps / (max_total_ms / 1e3)


def time_graph_step(dcp, dev, layers=4, reps=20):
    """Launch overhead of a whole decode step on the small sparse workload (16 rows, 64 heads,
    top-k 512, BF16, D = 4): `layers` fused calls, and the unfused form (one remap reused by
    every layer, then per layer partials + merge), eager vs replayed as one CUDA graph."""
    import synth
    g = synth.cfg2_sparse_topk512(device=dev)
    R, H, D, K = g.rows, g.heads, g.dcp, g.k
    out = torch.empty((R, H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((R, H), dtype=torch.float32, device=dev)
    loc = torch.empty((D, R, K), dtype=torch.int32, device=dev)
    cnt = torch.empty((D, R), dtype=torch.int32, device=dev)
    po = torch.empty((D, R, H, 512), dtype=torch.float32, device=dev)
    pl = torch.empty((D, R, H), dtype=torch.float32, device=dev)

    def ws_for(idx, count, o, l, n, fused):
        a = dcp._decode_args(g.q, g.pool, g.kv_dtype, g.block_table, g.row_seq, g.sm_scale, idx,
                             count, None, None, o, l, 0, False, None)
        return torch.zeros(dcp.mla_decode_workspace_size(a, n, fused) + 256, dtype=torch.uint8, device=dev)

    ws_f = ws_for(g.topk, None, out, lse, D, True)
    ws_p = ws_for(loc, cnt, po, pl, D, False)

    def fused():
        for _ in range(layers):
            dcp.mla_decode_dcp_fused(g.q, g.pool, g.kv_dtype, g.block_table, g.row_seq, g.sm_scale,
                                     D, g.interleave, idx=g.topk, out=out, lse=lse, workspace=ws_f)

    def unfused():
        dcp.dcp_remap_topk(g.topk, D, g.interleave, local_idx=loc, count=cnt)
        for _ in range(layers):
            dcp.mla_decode_partial_lse(g.q, g.pool, g.kv_dtype, g.block_table, g.row_seq, g.sm_scale,
                                       idx=loc, count=cnt, num_shards=D, out=po, lse=pl, workspace=ws_p)
            dcp.dcp_lse_merge(po, pl, out=out, lse=lse)

    res = {"workload": "sparse top-k 512, 64 heads, BF16 KV, 16 rows, DCP=4, %d layers per step" % layers}
    for name, fn in (("fused", fused), ("unfused", unfused)):
        fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        b.synchronize()
        eager = a.elapsed_time(b) / reps
        graph = torch.cuda.CUDAGraph()
        st = torch.cuda.Stream(dev)
        st.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(st):
            with torch.cuda.graph(graph, stream=st):
                fn()
        torch.cuda.current_stream(dev).wait_stream(st)
        graph.replay()
        torch.cuda.synchronize()
        a.record()
        for _ in range(reps):
            graph.replay()
        b.record()
        b.synchronize()
        res[name] = {"eager_us_per_layer": 1e3 * eager / layers,
                     "graph_us_per_layer": 1e3 * a.elapsed_time(b) / reps / layers}
    return res


def cpu_baseline_sample(prob):
    """Oracle timed on host cores on a bounded sample of the same workload (rank 0, N = 1)."""
    import oracle
    host = host_copy(prob)
    n = time_oracle_rows(host, 15.0)
    t0 = time.perf_counter()
    oracle.attention_problem(host, rows=list(range(n)))
    dt = time.perf_counter() - t0
    return {"value": n / dt, "unit": "rows/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": "%d of the 384 decode rows (2048 FP8 slots x 128 heads each), %.1f s"
                      % (n, dt)}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--seqs", type=int, default=64,
                    help="sequences of the workload (64 = the full workload; fewer only for "
                         "profiling captures that must stay small)")
    ap.add_argument("--kernel-path", default="auto", choices=["auto", "cuda_cores"],
                    help="decode kernel choice passed to every decode call (cuda_cores: the "
                         "CUDA-core kernel for every head count, for profiling it)")
    ap.add_argument("--kvwrite-only", action="store_true",
                    help="time only the DCP KV-cache write (for profiling its kernel) and print "
                         "its measurement")
    ap.add_argument("--topk-only", action="store_true",
                    help="time only the DSA top-k producer (for profiling its kernels) and "
                         "print its measurement")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import decode_context_sparse_gb300 as dcp
    from decode_context_sparse_gb300 import build
    build.build()
    dcp.load()

    peaks = load_peaks()
    if args.kvwrite_only:
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        res = time_kv_cache_write(dcp, dev, peaks, torch.cuda.current_stream(dev), flush,
                                  max(3, args.steps))
        print(json.dumps({"kv_cache_write": res}), flush=True)
        return
    if args.topk_only:
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        res = time_topk_producer(dcp, dev, peaks, torch.cuda.current_stream(dev), flush,
                                 max(3, args.steps), seqs=args.seqs)
        print(json.dumps({"topk_producer": res}), flush=True)
        return
    prob = make_workload(dev, args.seqs)
    kv_bytes, flops, valid = algorithmic(prob)
    R = prob.rows
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    out = torch.empty((R, prob.heads, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((R, prob.heads), dtype=torch.float32, device=dev)

    kpath = dcp.DCP_PATH_CUDA_CORES if args.kernel_path == "cuda_cores" else dcp.DCP_PATH_AUTO

    def step():
        dcp.mla_decode_dcp_fused(prob.q, prob.pool, prob.kv_dtype, prob.block_table, prob.row_seq,
                                 prob.sm_scale, prob.dcp, prob.interleave, idx=prob.topk,
                                 out=out, lse=lse, kernel_path=kpath)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()

    sampler = ClockSampler(dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    torch.cuda.synchronize()
    sampler.start()
    for i in range(args.steps):
        flush.fill_(i & 0xff)
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    times_ms = [a.elapsed_time(b) for a, b in evs]
    total_ms = max_over_ranks(sum(times_ms), dev)
    avg_ms = total_ms / args.steps
    value = whole_job_rate(R, args.steps, total_ms, ws)

    # unfused pipeline (remap -> partials -> merge), same workload, same timing rules
    D = prob.dcp
    loc = torch.empty((D, R, prob.k), dtype=torch.int32, device=dev)
    cnt = torch.empty((D, R), dtype=torch.int32, device=dev)
    po = torch.empty((D, R, prob.heads, 512), dtype=torch.float32, device=dev)
    pl = torch.empty((D, R, prob.heads), dtype=torch.float32, device=dev)

    def unfused():
        dcp.dcp_remap_topk(prob.topk, D, prob.interleave, local_idx=loc, count=cnt)
        dcp.mla_decode_partial_lse(prob.q, prob.pool, prob.kv_dtype, prob.block_table,
                                   prob.row_seq, prob.sm_scale, idx=loc, count=cnt, num_shards=D,
                                   out=po, lse=pl, kernel_path=kpath)
        dcp.dcp_lse_merge(po, pl, out=out, lse=lse)

    for _ in range(3):
        unfused()
    uev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(max(3, args.steps // 2))]
    for a, b in uev:
        flush.fill_(1)
        a.record(stream)
        unfused()
        b.record(stream)
    torch.cuda.synchronize()
    unfused_ms = statistics.mean(a.elapsed_time(b) for a, b in uev)
    kvw = time_kv_cache_write(dcp, dev, peaks, stream, flush, args.steps)
    topk_prod = time_topk_producer(dcp, dev, peaks, stream, flush, args.steps)
    prefill = time_prefill_chunk(dcp, dev, peaks, stream, flush, args.steps)
    graph_step = time_graph_step(dcp, dev)
    configs = time_configs(dcp, dev, peaks, stream, flush, args.steps)

    # end to end through the public API with host buffers: H2D of the step's inputs (queries,
    # top-k ids, row map, block tables) from pinned memory, D2H of the outputs
    h_q = prob.q.cpu().pin_memory()
    h_topk = prob.topk.cpu().pin_memory()
    h_rs = prob.row_seq.cpu().pin_memory()
    h_bt = prob.block_table.cpu().pin_memory()
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h_lse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    d_q, d_topk = torch.empty_like(prob.q), torch.empty_like(prob.topk)
    d_rs, d_bt = torch.empty_like(prob.row_seq), torch.empty_like(prob.block_table)

    def e2e_step():
        d_q.copy_(h_q, non_blocking=True)
        d_topk.copy_(h_topk, non_blocking=True)
        d_rs.copy_(h_rs, non_blocking=True)
        d_bt.copy_(h_bt, non_blocking=True)
        dcp.mla_decode_dcp_fused(d_q, prob.pool, prob.kv_dtype, d_bt, d_rs, prob.sm_scale,
                                 prob.dcp, prob.interleave, idx=d_topk, out=out, lse=lse)
        h_out.copy_(out, non_blocking=True)
        h_lse.copy_(lse, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e2e_ms = []
    for _ in range(args.steps):
        flush.fill_(2)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        e2e_step()
        b.record(stream)
        b.synchronize()
        e2e_ms.append(a.elapsed_time(b))
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_topk, h_rs, h_bt))
    d2h = h_out.numel() * h_out.element_size() + h_lse.numel() * h_lse.element_size()
    serial_ms = statistics.mean(e2e_ms)

    # the same steps pipelined as a serving loop runs them: step i's uploads (copy stream)
    # overlap step i-1's decode and step i-2's download (a third stream); two sets of device
    # buffers; every step still uploads its inputs from pinned host memory and downloads its
    # outputs.  (The 516 MB of KV each step gathers exceed L2, so no flush between steps.)
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    sets = [dict(q=torch.empty_like(prob.q), topk=torch.empty_like(prob.topk),
                 rs=torch.empty_like(prob.row_seq), bt=torch.empty_like(prob.block_table),
                 out=torch.empty_like(out), lse=torch.empty_like(lse),
                 h_out=torch.empty(out.shape, dtype=out.dtype).pin_memory(),
                 h_lse=torch.empty(lse.shape, dtype=lse.dtype).pin_memory()) for _ in range(2)]
    ev_up = [torch.cuda.Event() for _ in range(2)]
    ev_dec = [torch.cuda.Event() for _ in range(2)]
    ev_down = [torch.cuda.Event() for _ in range(2)]

    def pipelined(nsteps):
        for i in range(nsteps):
            b = sets[i % 2]
            with torch.cuda.stream(up):
                if i >= 2:
                    up.wait_event(ev_dec[i % 2])  # step i-2's decode has read these inputs
                b["q"].copy_(h_q, non_blocking=True)
                b["topk"].copy_(h_topk, non_blocking=True)
                b["rs"].copy_(h_rs, non_blocking=True)
                b["bt"].copy_(h_bt, non_blocking=True)
                ev_up[i % 2].record(up)
            stream.wait_event(ev_up[i % 2])
            if i >= 2:
                stream.wait_event(ev_down[i % 2])  # step i-2's download has read these outputs
            dcp.mla_decode_dcp_fused(b["q"], prob.pool, prob.kv_dtype, b["bt"], b["rs"],
                                     prob.sm_scale, prob.dcp, prob.interleave, idx=b["topk"],
                                     out=b["out"], lse=b["lse"])
            ev_dec[i % 2].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(ev_dec[i % 2])
                b["h_out"].copy_(b["out"], non_blocking=True)
                b["h_lse"].copy_(b["lse"], non_blocking=True)
                ev_down[i % 2].record(down)

    pipelined(4)
    torch.cuda.synchronize()
    t_a, t_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_a.record(stream)
    up.wait_stream(stream)
    pipelined(args.steps)
    stream.wait_stream(down)
    stream.wait_stream(up)
    t_b.record(stream)
    torch.cuda.synchronize()
    pipe_ms = max_over_ranks(t_a.elapsed_time(t_b), dev)
    e2e_val = whole_job_rate(R, args.steps, pipe_ms, ws)

    if rank != 0:
        if ws > 1:
            torch.distributed.destroy_process_group()
        return

    t_s = avg_ms / 1e3
    hbm_tbs = kv_bytes / t_s / 1e12
    tflops = flops / t_s / 1e12
    t_hbm = kv_bytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops / (peaks["bf16_tflops"] * 1e12)
    bound = "tensor" if t_tc >= t_hbm else "hbm"
    if bound == "tensor":
        roof = {"bound": "tensor", "achieved": tflops, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": tflops / peaks["bf16_tflops"]}
    else:
        roof = {"bound": "hbm", "achieved": hbm_tbs * 1e3, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": hbm_tbs * 1e3 / peaks["hbm_gbs"]}
    # traffic: the ncu capture's DRAM bytes per row times the rows of this launch (not
    # measured in this run; see TRAFFIC_CAPTURE), beside the algorithmic bytes it compares to
    alg_all = kv_bytes + prob.q.numel() * 2 + out.numel() * 2 + lse.numel() * 4 + \
        prob.topk.numel() * 4
    traffic = TRAFFIC_CAPTURE["bytes_per_row"] * R if prob.heads == 128 else None
    roof["traffic"] = traffic
    roof["traffic_unit"] = "bytes"
    roof["traffic_src"] = ("ncu capture of %s on a %d-row slice of this workload, scaled to %d "
                           "rows" % (TRAFFIC_CAPTURE["kernel"], TRAFFIC_CAPTURE["rows"], R))
    roof["algorithmic_bytes_kv"] = kv_bytes
    roof["algorithmic_bytes_all"] = alg_all
    if traffic is not None:
        roof["traffic_over_kv"] = traffic / kv_bytes
        roof["traffic_over_all"] = traffic / alg_all
    roof["peak_src"] = peaks["src"]
    # the tensor-core kernel multiplies FP16 operands (fp32 accumulation), whose dense rate
    # is the bf16 one, so the measured bf16 burst peak is the FP16 peak (nominal ratio 1)
    roof["peak_dtype"] = "fp16 operands: the measured bf16 burst peak x 1 (same nominal rate)"
    roof["kernel"] = "mla_decode_dcp_fused"
    roof["roofline_us"] = 1e6 * max(t_hbm, t_tc)
    line = {
        "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": ws, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": avg_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "rows": R, "heads": prob.heads, "topk": prob.k,
                   "dcp": prob.dcp, "interleave": prob.interleave, "context": 131072,
                   "kv_dtype": "fp8_e4m3_per128_scale", "l2": "flushed between steps (256 MB write)",
                   "arithmetic": "FP16 tensor-core operands, fp32 accumulation and softmax, "
                                 "BF16 output",
                   "parallelism": "replicas" if ws > 1 else "single GPU"},
        "achieved_hbm_tbs": hbm_tbs,
        "achieved_tflops": tflops,
        "tokens_per_s": value,
        "kv_slots_gathered_per_s": ws * valid * args.steps / (total_ms / 1e3),
        "us_per_layer": 1e3 * avg_ms,
        "unfused": {"ms_per_step": unfused_ms, "rows_per_s": R / (unfused_ms / 1e3),
                    "launches_per_step": 3},
        "roofline": roof,
        "kv_cache_write": kvw,
        "topk_producer": topk_prod,
        "prefill_chunk": prefill,
        "graph_step": graph_step,
        "configs": configs,
        "clocks": clocks,
        "e2e": {"value": e2e_val, "unit": "rows/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": pipe_ms / args.steps,
                "pipelined": "uploads, decode and downloads of consecutive steps on 3 streams",
                "serial_ms_per_step": serial_ms},
        # per fused call: the persistent decode and the merge of rows cut between CTA pairs
        "gpu_launches": 2 * args.steps,
    }
    if ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_sample(prob)
    print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
