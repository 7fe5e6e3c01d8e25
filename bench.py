"""Benchmark of the DSA indexer hot path on one GB300 (or N replicas under torchrun).

One step = one full pass of the indexer over one synthetic batch: q-k scoring on
the tensor cores with the fused ReLU / head-weighted reduction / causal mask, then
the per-row top-k.  Default workload: prefill of one 8192-token sequence, causal,
H=64 indexer heads, D=128, index_topk=2048, bf16 q/k, fp32 w ~ N(0,1)/8.

Prints ONE JSON line (rank 0).  `value` counts causal query-key pairs scored per
second (each pair covers all H heads), whole job, inputs resident in HBM; `e2e`
is the same metric through the public API with pinned host buffers copied in and
the top-k copied out inside the timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

`--impl reference` times the CPU oracle (test infrastructure, fp64, full sort)
on the host cores on a bounded sample of query rows of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = ("indexer query-key scores/sec + top-k rows/sec; % of TC peak (prefill), "
          "% HBM BW (decode)")
UNIT = "scores/s"
WORKLOAD = "prefill T=S=8192 causal, H=64, D=128, index_topk=2048, bf16 q/k, fp32 w"
T = S = 8192
H, D, TOPK = 64, 128, 2048
PAIRS = T * (T + 1) // 2                     # causal (t, s) pairs, each over all H heads
FLOPS = 2 * H * D * PAIRS                    # tensor-core flops of the q.k contraction


def _env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


E2E_CHUNK = int(os.environ.get("DSA_BENCH_E2E_CHUNK", "0"))  # query rows per transfer chunk (0: library default)


def kernel_source_hash():
    h = hashlib.sha256()
    for f in ("score_tc.cu", "ptx.cuh", "internal.h"):
        with open(os.path.join(ROOT, "sparse_attention_token_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic():
    """DRAM bytes per score-kernel launch from the committed ncu summary, if it was
    taken on the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "score_kernel_prefill_8k.json")
    if not os.path.exists(p):
        return None
    try:
        with open(p) as f:
            d = json.load(f)
        if d.get("kernel_source_hash") != kernel_source_hash():
            return None
        return d.get("dram_bytes_per_launch_full_size")
    except Exception:
        return None


def measure_tensor_peaks(dev, n: int = 8192, reps: int = 10):
    """Dense tensor-core throughput of this GPU measured in this run: bf16 torch.matmul and
    e4m3 torch._scaled_mm (per-tensor scales, bf16 out) at n^3, best of `reps` (CUDA events).
    The e4m3 figure is the roofline peak of the FP8 score kernel."""
    g = torch.Generator(device=dev)
    g.manual_seed(11)
    a = torch.randn((n, n), generator=g, device=dev).to(torch.bfloat16)
    b = torch.randn((n, n), generator=g, device=dev).to(torch.bfloat16)
    out = {}

    def best(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize(dev)
        t = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize(dev)
            t.append(e0.elapsed_time(e1))
        return 2.0 * n ** 3 / (min(t) / 1e3) / 1e12

    out["bf16_tflops"] = best(lambda: torch.matmul(a, b))
    a8 = a.to(torch.float8_e4m3fn)
    b8 = b.to(torch.float8_e4m3fn).t().contiguous().t()   # column-major second operand
    one = torch.ones((), dtype=torch.float32, device=dev)
    try:
        out["e4m3_tflops"] = best(lambda: torch._scaled_mm(a8, b8, scale_a=one, scale_b=one,
                                                           out_dtype=torch.bfloat16))
    except Exception as exc:  # noqa: BLE001 -- reported, not hidden
        out["e4m3_tflops"] = None
        out["e4m3_error"] = str(exc).splitlines()[0][:200]
    out["how"] = (f"{n}^3, best of {reps}, CUDA events: torch.matmul bf16; torch._scaled_mm e4m3 x e4m3 "
                  "with per-tensor fp32 scales, bf16 out")
    del a, b, a8, b8
    torch.cuda.empty_cache()
    return out


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons in the background."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        rows = self._rows()
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        inside = [r for r in rows if t0 - 0.02 <= r[0] <= t1 + 0.02]
        window = "timed region"
        if not inside:
            inside = sorted(rows, key=lambda r: min(abs(r[0] - t0), abs(r[0] - t1)))[:3]
            window = "nearest samples (timed region shorter than the sampling period)"
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside), "window": window}

    def _rows(self):
        if getattr(self, "_cache", None) is not None:
            return self._cache
        rows = []
        if self.path and os.path.exists(self.path):
            for line in open(self.path):
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    frac = float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                    rows.append((ts + frac, float(parts[1]), float(parts[2]), parts[5:9]))
                except Exception:
                    continue
            os.unlink(self.path)
        self._cache = rows
        return rows


def make_inputs(seed: int = 0):
    import workloads
    return workloads.prefill_8k(seed=seed)


def sm_clock_in_band(a, b):
    """Average SM clock of every SM over the timed region: (cycle counter after - before) /
    (global ns timer after - before) per SM, from two samples on the launch stream that
    bracket the region (one-thread blocks, a few per SM)."""
    first, last = {}, {}
    for row in a.tolist():
        sm, c, t = row
        if sm not in first or t < first[sm][1]:
            first[sm] = (c, t)
    for row in b.tolist():
        sm, c, t = row
        if sm not in last or t > last[sm][1]:
            last[sm] = (c, t)
    mhz = sorted(1e3 * (last[s][0] - first[s][0]) / (last[s][1] - first[s][1])
                 for s in first if s in last and last[s][1] > first[s][1])
    if not mhz:
        return None
    return {"sm_mhz_mean": sum(mhz) / len(mhz), "sm_mhz_min": mhz[0], "sm_mhz_max": mhz[-1], "sms": len(mhz),
            "how": "cycle counter and global ns timer read on every SM just before and just after the timed "
                   "region (dsa_clock_sample on the launch stream)"}


def run_ours(args, rank: int, world: int, local_rank: int):
    import sparse_attention_token_gb300 as dsa
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    case = make_inputs(seed=rank)
    q, k, w = case.q.to(dev), case.k.to(dev), case.w.to(dev)
    ld = S
    scores = torch.empty((T, ld), dtype=torch.float32, device=dev)
    topk = torch.empty((T, TOPK), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        dsa.dsa_indexer_scores(q, k, w, q_pos0=0, scores=scores, stream=stream)
        dsa.dsa_indexer_topk(scores, T=T, S=S, q_pos0=0, topk_limit=TOPK, topk=topk, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if dsa.dsa_check_device_status(stream) != dsa.DSA_OK:
        raise RuntimeError("device status error during warm-up")

    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)

    # ---- timed region: K steps, inputs resident; per-kernel events on the launch stream
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    n_probe = 4 * torch.cuda.get_device_properties(dev).multi_processor_count
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    clk0 = dsa.dsa_clock_sample(n_probe, stream)  # just outside the timed region, same stream
    start.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        dsa.dsa_indexer_scores(q, k, w, q_pos0=0, scores=scores, stream=stream)
        ev[i][1].record(stream)
        dsa.dsa_indexer_topk(scores, T=T, S=S, q_pos0=0, topk_limit=TOPK, topk=topk, stream=stream)
        ev[i][2].record(stream)
    end.record(stream)
    clk1 = dsa.dsa_clock_sample(n_probe, stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    total_ms = start.elapsed_time(end)
    score_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / args.steps
    topk_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / args.steps
    status = dsa.dsa_check_device_status(stream)

    # ---- end to end through the public API: pinned host in, top-k out, every step.
    # dsa_indexer_dense_host copies the query rows in chunk by chunk and each chunk's top-k
    # rows back, overlapped with the kernels of other chunks.
    q_h = case.q.pin_memory()
    k_h = case.k.pin_memory()
    w_h = case.w.pin_memory()
    topk_h = torch.empty((T, TOPK), dtype=torch.int32).pin_memory()
    del scores, topk
    torch.cuda.empty_cache()
    ws = torch.empty(dsa.dsa_indexer_dense_host_workspace_size(T, S, H, D, dsa.DSA_BF16, TOPK, E2E_CHUNK),
                     dtype=torch.uint8, device=dev)
    e2e_call = lambda: dsa.dsa_indexer_dense_host(q_h, k_h, w_h, q_pos0=0, topk_limit=TOPK, chunk_rows=E2E_CHUNK,
                                                  topk=topk_h, workspace=ws, stream=stream)
    e2e_steps = max(1, min(args.steps, 50))
    for _ in range(2):
        e2e_call()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_call()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    t_wall2 = time.time()
    sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall1)
    clocks["in_band"] = sm_clock_in_band(clk0.cpu(), clk1.cpu())
    # the timed region is short next to the sampling period: also report the samples
    # over the timed region and the end-to-end loop that follows it
    clocks_e2e = sampler.summary(t_wall0, t_wall2)
    clocks["timed_and_e2e"] = {k: clocks_e2e[k] for k in ("sm_mhz", "sm_max_mhz", "reasons", "samples")}
    h2d = q_h.numel() * q_h.element_size() + k_h.numel() * k_h.element_size() + w_h.numel() * w_h.element_size()
    d2h = topk_h.numel() * topk_h.element_size()

    total_ms, score_ms, topk_ms, e2e_ms = max_over_ranks([total_ms, score_ms, topk_ms, e2e_ms], world, dev)
    return dict(total_ms=total_ms, score_ms=score_ms, topk_ms=topk_ms, e2e_ms=e2e_ms, clocks=clocks,
                h2d=h2d, d2h=d2h, status=status, case=case, e2e_steps=e2e_steps)



def max_over_ranks(values, world: int, device) -> list:
    """Each timing's maximum over the ranks (the slowest replica sets the job's time)."""
    vals = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(vals, op=torch.distributed.ReduceOp.MAX)
    return vals.tolist()


def job_rate(units_per_rank: float, world: int, ms_per_step_max: float) -> float:
    """Whole-job throughput: the units every rank processed in one step, over the
    slowest rank's step time (weak scaling: each rank holds the same workload)."""
    return units_per_rank * world / (ms_per_step_max / 1e3)


# ----------------------------------------------------------------------------- other workloads
# Measured after the headline (same process, same GPU); inputs generated on the device
# with a seeded generator where they are large.

def _time_events(fn, iters, stream):
    for _ in range(2):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(iters):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / iters


def _paged_on_device(B, lens, q_len, H, D, page, q_fp8, k_fp8, seed, dev):
    """Seeded device-side paged case: N(0,1) keys (e4m3 with per-token amax/448 scales when
    k_fp8), q N(0,1) (e4m3 per (t,h) when q_fp8), w N(0,1)/8, pages in a random permutation."""
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    lens = [int(x) for x in lens]
    pages = [(L + page - 1) // page for L in lens]
    num_pages = sum(pages) + 1
    perm = torch.randperm(num_pages, generator=g, device=dev).to(torch.int32)
    mp = max(pages)
    bt = torch.full((B, mp), -1, dtype=torch.int32, device=dev)
    cur = 0
    for b, npg in enumerate(pages):
        bt[b, :npg] = perm[cur:cur + npg]
        cur += npg
    total_q = q_len * B
    kf = torch.randn((num_pages, page, D), generator=g, device=dev, dtype=torch.float32)
    qf = torch.randn((total_q, H, D), generator=g, device=dev, dtype=torch.float32)
    w = torch.randn((total_q, H), generator=g, device=dev, dtype=torch.float32) / 8.0

    def quant(x):
        amax = x.abs().amax(dim=-1, keepdim=True)
        sc = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
        return (x / sc).to(torch.float8_e4m3fn), sc.squeeze(-1).contiguous()

    k_cache, k_scale = quant(kf) if k_fp8 else (kf.to(torch.bfloat16), None)
    q, q_scale = quant(qf) if q_fp8 else (qf.to(torch.bfloat16), None)
    del kf, qf
    cu = torch.arange(0, total_q + 1, q_len, dtype=torch.int32, device=dev)
    seq = torch.tensor(lens, dtype=torch.int32, device=dev)
    return dict(q=q, q_scale=q_scale, w=w, k_cache=k_cache, k_scale_cache=k_scale, cu_q_lens=cu, seq_lens=seq,
                block_tables=bt, max_seq_len=max(lens))


def _chunked_prefill_fp8(dev, stream, peaks, iters=3):
    """8192 queries at 57344..65535 vs a 65536-key cache, e4m3 q and k (one dsa_indexer call)."""
    import ctypes
    import sparse_attention_token_gb300 as dsa
    bf16_peak = float(peaks["bf16_tflops"])
    e4m3_peak = peaks.get("e4m3_tflops")
    c = _paged_on_device(1, [65536], 8192, 64, 128, 64, True, True, 4, dev)
    args, keep = dsa.make_indexer_args(c["q"], c["w"], c["k_cache"], c["cu_q_lens"], c["seq_lens"],
                                       c["block_tables"], max_seq_len=c["max_seq_len"], topk_limit=2048,
                                       q_scale=c["q_scale"], k_scale_cache=c["k_scale_cache"])
    L = dsa.lib()
    ms = _time_events(lambda: L.dsa_indexer(ctypes.byref(args), stream.cuda_stream), iters, stream)
    pairs = sum(57344 + i + 1 for i in range(8192))
    flops = 2 * 64 * 128 * pairs
    out = {
        "workload": "8192 queries at 57344..65535 vs a 65536-key paged cache (page 64), e4m3 q/k with fp32 scales, "
                    "H=64, D=128, index_topk=2048",
        "ms_per_step": ms, "scores_per_s": pairs / (ms / 1e3), "topk_rows_per_s": 8192 / (ms / 1e3),
        "tflops_step": flops / (ms / 1e3) / 1e12}
    if e4m3_peak:
        out["tc_frac_step"] = out["tflops_step"] / e4m3_peak
        out["peak"] = f"e4m3 dense measured in this run (torch._scaled_mm 8192^3): {e4m3_peak:.0f} TFLOP/s"
    else:
        out["tc_frac_step"] = out["tflops_step"] / (2 * bf16_peak)
        out["peak"] = f"e4m3 dense = 2 x measured bf16 ({2 * bf16_peak:.0f} TFLOP/s, nominal ratio)"
    del c, args, keep
    torch.cuda.empty_cache()
    return out


def _decode_b64_fp8_cache(dev, stream, peaks, iters=10):
    """Decode B=64, contexts U[4096, 65536], bf16 q against a paged e4m3 cache."""
    import ctypes
    import sparse_attention_token_gb300 as dsa
    import workloads
    hbm = float(peaks["hbm_gbs"])
    lens = workloads.decode_lens(64, 4096, 65536, 0)
    page = _env_int("DSA_BENCH_DECODE_PAGE", 64)  # another page size only for the page-size study
    c = _paged_on_device(64, lens, 1, 64, 128, page, False, True, 5, dev)
    args, keep = dsa.make_indexer_args(c["q"], c["w"], c["k_cache"], c["cu_q_lens"], c["seq_lens"],
                                       c["block_tables"], max_seq_len=c["max_seq_len"], topk_limit=2048,
                                       k_scale_cache=c["k_scale_cache"])
    L = dsa.lib()
    rc = L.dsa_indexer(ctypes.byref(args), stream.cuda_stream)
    if rc != 0:
        raise RuntimeError(f"dsa_indexer (bf16 q, e4m3 cache): {dsa.dsa_status_string(rc)}")
    ms = _time_events(lambda: L.dsa_indexer(ctypes.byref(args), stream.cuda_stream), iters, stream)
    keys = sum(lens)
    # algorithmic bytes: e4m3 keys + fp32 key scales + page ids + q + w + int32 top-k out
    dec_bytes = keys * (128 + 4) + sum((x + page - 1) // page for x in lens) * 4 + 64 * 64 * 128 * 2 + 64 * 64 * 4 \
        + 64 * 2048 * 4
    out = {
        "workload": "decode B=64, one query per sequence, contexts U[4096, 65536] (seeded), bf16 q, "
                    f"paged e4m3 cache (page {page}) with fp32 per-token scales, H=64, D=128, index_topk=2048",
        "ms_per_step": ms, "keys_per_s": keys / (ms / 1e3), "keys": keys,
        "algorithmic_bytes": dec_bytes, "hbm_gbs": dec_bytes / (ms / 1e3) / 1e9,
        "hbm_frac": dec_bytes / (ms / 1e3) / 1e9 / hbm,
        "note": "includes the fp32 score round trip (4 B written + 4 B read per key) that is not in the "
                "algorithmic bytes"}
    del c, args, keep
    torch.cuda.empty_cache()
    return out


def _indexshare_stack(dev, stream, peaks, iters=5):
    """12 layers [full, shared, shared] x 4, decode B=32 at 32768 keys, bf16 caches."""
    import ctypes
    import sparse_attention_token_gb300 as dsa
    hbm = float(peaks["hbm_gbs"])
    types = ["full", "shared", "shared"] * 4
    fulls, keeps = [], []
    for li in range(4):
        c = _paged_on_device(32, [32768] * 32, 1, 64, 128, 64, False, False, 100 + li, dev)
        a, k2 = dsa.make_indexer_args(c["q"], c["w"], c["k_cache"], c["cu_q_lens"], c["seq_lens"],
                                      c["block_tables"], max_seq_len=c["max_seq_len"], topk_limit=2048)
        fulls.append(a)
        keeps.append((c, k2))
    layer_args = []
    fi = 0
    for t in types:
        if t == "full":
            layer_args.append(fulls[fi])
            fi += 1
        else:
            layer_args.append(None)
    L = dsa.lib()
    stack_ms = _time_events(lambda: dsa.dsa_indexer_stack(types, layer_args, stream=stream), iters, stream)
    allfull_ms = _time_events(lambda: [L.dsa_indexer(ctypes.byref(fulls[i % 4]), stream.cuda_stream)
                                       for i in range(12)], iters, stream)
    keys = 32 * 32768
    bytes_full = keys * 128 * 2 + 32 * 64 * 128 * 2 + 32 * 64 * 4 * 2 + 32 * 2048 * 4
    out = {
        "workload": "12 layers [full, shared, shared] x 4, decode B=32 at 32768 keys, bf16 paged caches "
                    "(one per full layer), H=64, D=128, index_topk=2048",
        "ms_stack": stack_ms, "ms_all_full": allfull_ms, "speedup_vs_all_full": allfull_ms / stack_ms,
        "full_layer_ms": stack_ms / 4,
        "hbm_gbs_full_layers": 4 * bytes_full / (stack_ms / 1e3) / 1e9,
        "hbm_frac_full_layers": 4 * bytes_full / (stack_ms / 1e3) / 1e9 / hbm,
        "bytes_per_full_layer": bytes_full}
    del keeps, fulls, layer_args
    torch.cuda.empty_cache()
    return out


def _cache_append_fp8(dev, stream, peaks, iters=20):
    """65536 new bf16 keys (D=128) quantised into a paged e4m3 cache through slot_mapping."""
    import sparse_attention_token_gb300 as dsa
    hbm = float(peaks["hbm_gbs"])
    g = torch.Generator(device=dev)
    g.manual_seed(6)
    n, PS = 65536, 64
    pages = n // PS + 8
    k_new = torch.randn((n, 128), generator=g, device=dev).to(torch.bfloat16)
    slots = torch.randperm(pages * PS, generator=g, device=dev)[:n].to(torch.int64)
    cache = torch.zeros((pages, PS, 128), dtype=torch.uint8, device=dev).view(torch.float8_e4m3fn)
    scales = torch.zeros((pages, PS), dtype=torch.float32, device=dev)
    ms = _time_events(lambda: dsa.dsa_indexer_cache_append(k_new, slots, cache, scales, stream=stream), iters, stream)
    nbytes = n * (128 * 2 + 8 + 128 + 4)  # bf16 row + slot read, codes + scale written
    out = {"workload": "65536 new keys, bf16 D=128, quantised per token into a paged e4m3 cache (page 64)",
           "ms_per_step": ms, "tokens_per_s": n / (ms / 1e3), "algorithmic_bytes": nbytes,
           "hbm_gbs": nbytes / (ms / 1e3) / 1e9, "hbm_frac": nbytes / (ms / 1e3) / 1e9 / hbm}
    del k_new, slots, cache, scales
    torch.cuda.empty_cache()
    return out


def _frontend_fp8(dev, stream, peaks, iters=20):
    """dsa_indexer_prepare on an e4m3 cache: 8192 prefill tokens and 64 decode tokens."""
    import ctypes
    import sparse_attention_token_gb300 as dsa
    import workloads
    bf16_peak, hbm = float(peaks["bf16_tflops"]), float(peaks["hbm_gbs"])
    Dm, R, H, D, r = 6144, 2048, 64, 128, 64
    out = {"workload": f"indexer front-end, e4m3 cache: hidden {Dm}, q_rank {R}, H={H}, D={D}, rope_dim={r} "
                       "(projection sizes assumed; the pages give none), synthetic N(0,1) activations"}
    for name, T in (("prefill_8k", 8192), ("decode_64", 64)):
        c = workloads.frontend_case(T, Dm, R, H, D, rope_dim=r, fp8=True, seed=7)
        to = lambda t: None if t is None else t.to(dev)
        a, keep, _ = dsa.make_prepare_args(to(c.hidden), to(c.qa_normed), to(c.rope_cos), to(c.rope_sin), to(c.wq_b),
                                           to(c.wk), to(c.weights_proj), to(c.k_norm_weight), to(c.k_cache),
                                           to(c.slot_mapping), H=H, rope_dim=r, k_scale_cache=to(c.k_scale_cache))
        L = dsa.lib()
        fn = lambda: L.dsa_indexer_prepare(ctypes.byref(a), stream.cuda_stream)
        if fn() != 0:
            raise RuntimeError("dsa_indexer_prepare failed")
        ms = _time_events(fn, iters, stream)
        # the same call captured once in a CUDA graph and replayed: the device time without
        # the host's per-call launch and GEMM-setup cost (how a serving step would run it)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            if L.dsa_indexer_prepare(ctypes.byref(a), torch.cuda.current_stream().cuda_stream) != 0:
                raise RuntimeError("dsa_indexer_prepare failed under capture")
        ms_graph = _time_events(graph.replay, iters, stream)
        flops = 2.0 * T * (R * H * D + Dm * D + Dm * H)
        wbytes = 2.0 * (H * D * R + D * Dm + H * Dm)
        out[name] = {"tokens": T, "ms_per_step": ms, "ms_per_step_graph": ms_graph,
                     "gemm_tflops": flops / (ms / 1e3) / 1e12, "tc_frac": flops / (ms / 1e3) / 1e12 / bf16_peak,
                     "weight_bytes_hbm_frac": wbytes / (ms / 1e3) / 1e9 / hbm,
                     "weight_bytes_hbm_frac_graph": wbytes / (ms_graph / 1e3) / 1e9 / hbm}
        del graph
        del a, keep, c
        torch.cuda.empty_cache()
    return out


def _key_sharded_prefill(dev, stream, peaks, iters=10):
    """The 8K prefill with its keys split into two shards, scored one after the other on this
    GPU (virtual shards): per-shard candidates, then the exact merge of both lists."""
    import ctypes
    import sparse_attention_token_gb300 as dsa
    hbm = float(peaks["hbm_gbs"])
    g = torch.Generator(device=dev)
    g.manual_seed(12)
    Tq, Sk, K, bounds = 8192, 8192, 2048, (0, 4096, 8192)
    q = torch.randn((Tq, H, D), generator=g, device=dev).to(torch.bfloat16)
    k = torch.randn((Sk, D), generator=g, device=dev).to(torch.bfloat16)
    w = torch.randn((Tq, H), generator=g, device=dev) / 8.0
    ns = len(bounds) - 1
    ci = torch.empty((ns, Tq, K), dtype=torch.int32, device=dev)
    cs = torch.empty((ns, Tq, K), dtype=torch.float32, device=dev)
    topk = torch.empty((Tq, K), dtype=torch.int32, device=dev)
    nb = ctypes.c_size_t(0)
    L = dsa.lib()
    L.dsa_indexer_shard_candidates_workspace_size(Tq, max(b1 - b0 for b0, b1 in zip(bounds[:-1], bounds[1:])),
                                                  ctypes.byref(nb))
    ws = torch.empty(nb.value, dtype=torch.uint8, device=dev)
    shards = [k[b0:b1].contiguous() for b0, b1 in zip(bounds[:-1], bounds[1:])]

    def candidates():
        for j, (b0, b1) in enumerate(zip(bounds[:-1], bounds[1:])):
            rc = L.dsa_indexer_shard_candidates(q.data_ptr(), 0, None, shards[j].data_ptr(), 0, None, w.data_ptr(),
                                                Tq, b1 - b0, H, D, 0, b0, K, ci[j].data_ptr(), cs[j].data_ptr(),
                                                ws.data_ptr(), ws.numel(), stream.cuda_stream)
            if rc != 0:
                raise RuntimeError(dsa.dsa_status_string(rc))

    def merge():
        rc = L.dsa_indexer_merge_candidates(cs.data_ptr(), ci.data_ptr(), ns, Tq, K, K, K, 0, topk.data_ptr(),
                                            stream.cuda_stream)
        if rc != 0:
            raise RuntimeError(dsa.dsa_status_string(rc))

    ms_cand = _time_events(candidates, iters, stream)
    ms_merge = _time_events(merge, iters, stream)
    ms_all = _time_events(lambda: (candidates(), merge()), iters, stream)
    merge_bytes = ns * Tq * K * 8 + Tq * K * 4   # candidate indices and scores in, top-k out
    out = {"workload": "prefill T=S=8192 causal, H=64, D=128, index_topk=2048, bf16, keys in 2 shards "
                       "(0..4095, 4096..8191) scored one after the other on this GPU, then merged",
           "ms_per_step": ms_all, "ms_candidates": ms_cand, "ms_merge": ms_merge,
           "scores_per_s": PAIRS / (ms_all / 1e3),
           "merge_hbm_gbs": merge_bytes / (ms_merge / 1e3) / 1e9,
           "merge_hbm_frac": merge_bytes / (ms_merge / 1e3) / 1e9 / hbm}
    del q, k, w, ci, cs, topk, ws, shards
    torch.cuda.empty_cache()
    return out


def _sparse_mla_decode(dev, stream, peaks, iters=10):
    """Sparse MLA after the indexer: decode B=64, one query per sequence, contexts U[4096, 65536],
    64 heads, 2048 selected keys per query, bf16 latent cache (kv_rank 512, rope 64, page 64)."""
    import ctypes
    import sparse_attention_token_gb300 as dsa
    import workloads
    hbm = float(peaks["hbm_gbs"])
    g = torch.Generator(device=dev)
    g.manual_seed(13)
    B = _env_int("DSA_BENCH_MLA_BATCH", 64)  # a smaller batch only for profiler captures
    Hh, K, page, R, rd = 64, 2048, 64, 512, 64
    lens = workloads.decode_lens(B, 4096, 65536, 0)
    pages = [(L + page - 1) // page for L in lens]
    num_pages = sum(pages) + 1
    perm = torch.randperm(num_pages, generator=g, device=dev).to(torch.int32)
    bt = torch.full((B, max(pages)), -1, dtype=torch.int32, device=dev)
    cur = 0
    for b, npg in enumerate(pages):
        bt[b, :npg] = perm[cur:cur + npg]
        cur += npg
    cache_c = torch.randn((num_pages, page, R), generator=g, device=dev).to(torch.bfloat16)
    cache_r = torch.randn((num_pages, page, rd), generator=g, device=dev).to(torch.bfloat16)
    q_nope = torch.randn((B, Hh, R), generator=g, device=dev).to(torch.bfloat16)
    q_rope = torch.randn((B, Hh, rd), generator=g, device=dev).to(torch.bfloat16)
    # each query's selection: 2048 distinct positions of its context, in random order
    topk = torch.stack([torch.randperm(L, generator=g, device=dev)[:K] for L in lens]).to(torch.int32)
    cu = torch.arange(0, B + 1, dtype=torch.int32, device=dev)
    seq = torch.tensor(lens, dtype=torch.int32, device=dev)
    a, keep = dsa.make_sparse_mla_args(q_nope, q_rope, cache_c, cache_r, bt, cu, seq, topk,
                                       scale=1.0 / (R + rd) ** 0.5)
    L = dsa.lib()
    rc = L.dsa_sparse_mla(ctypes.byref(a), stream.cuda_stream)
    if rc != 0:
        raise RuntimeError(f"dsa_sparse_mla: {dsa.dsa_status_string(rc)}")
    ms = _time_events(lambda: L.dsa_sparse_mla(ctypes.byref(a), stream.cuda_stream), iters, stream)
    # algorithmic bytes: the selected latent rows, q, the selection and the fp32 output
    nbytes = B * K * (R + rd) * 2 + B * Hh * (R + rd) * 2 + B * K * 4 + B * Hh * R * 4
    flops = 2.0 * B * Hh * K * (R + rd + R)
    out = {"workload": f"sparse MLA decode B={B}, one query per sequence, contexts U[4096, 65536], 64 heads, "
                       "2048 selected keys per query, bf16 latent cache (kv_rank 512, rope 64, page 64)",
           "ms_per_step": ms, "queries_per_s": B / (ms / 1e3), "algorithmic_bytes": nbytes,
           "hbm_gbs": nbytes / (ms / 1e3) / 1e9, "hbm_frac": nbytes / (ms / 1e3) / 1e9 / hbm,
           "tflops": flops / (ms / 1e3) / 1e12}
    del a, keep, cache_c, cache_r, q_nope, q_rope, topk
    torch.cuda.empty_cache()
    return out


OTHER_WORKLOADS = {
    "frontend_fp8": _frontend_fp8,
    "cache_append_fp8": _cache_append_fp8,
    "chunked_prefill_fp8": _chunked_prefill_fp8,
    "decode_b64_fp8_cache": _decode_b64_fp8_cache,
    "indexshare_stack": _indexshare_stack,
    "key_sharded_prefill": _key_sharded_prefill,
    "sparse_mla_decode": _sparse_mla_decode,
}


def run_other_workloads(dev, stream, peaks):
    return {name: fn(dev, stream, peaks) for name, fn in OTHER_WORKLOADS.items()}


def cpu_sample_rows(n_rows: int):
    """Stratified sample of query rows (positions spread over the sequence, first and last included)."""
    if n_rows >= T:
        return list(range(T))
    step = (T - 1) / (n_rows - 1)
    return sorted({int(round(i * step)) for i in range(n_rows)})


def time_oracle(case, rows, n_threads=0):
    import oracle
    t0 = time.perf_counter()
    oracle.dense(case.q, case.k, case.w, T=case.T, S=case.S, H=case.H, D=case.D, q_pos0=0,
                 topk_limit=TOPK, k_out=TOPK, rows=rows, n_threads=n_threads)
    dt = time.perf_counter() - t0
    pairs = sum(r + 1 for r in rows)
    return pairs / dt, dt, pairs


def cpu_baseline(case, budget_s: float = 15.0):
    import oracle
    cores = oracle.max_threads()
    rows = cpu_sample_rows(16)
    rate, dt, pairs = time_oracle(case, rows)
    # grow the sample to roughly the budget
    n = int(min(T, max(16, 16 * budget_s / max(dt, 1e-3))))
    if n > 16:
        rows = cpu_sample_rows(n)
        rate, dt, pairs = time_oracle(case, rows)
    return {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{len(rows)} query rows stratified over positions 0..{T - 1} of the same workload "
                      f"({pairs} causal pairs, {dt:.1f} s); fp64, full sort per row"}


def run_reference(args):
    case = make_inputs(seed=0)
    import oracle
    cores = oracle.max_threads()
    # size a step so that warm-up + K steps finish within ~3 minutes
    probe_rows = cpu_sample_rows(8)
    _, dt_probe, _ = time_oracle(case, probe_rows)
    per_row = dt_probe / len(probe_rows)
    total_steps = max(1, args.steps + args.warmup)
    rows_per_step = int(max(2, min(256, 150.0 / total_steps / max(per_row, 1e-4))))
    rows = cpu_sample_rows(rows_per_step)
    for _ in range(args.warmup):
        time_oracle(case, rows)
    t0 = time.perf_counter()
    pairs = 0
    for _ in range(args.steps):
        _, _, p = time_oracle(case, rows)
        pairs += p
    dt = time.perf_counter() - t0
    value = pairs / dt
    sample = (f"{len(rows)} query rows per step, stratified over positions 0..{T - 1} "
              f"({pairs // max(args.steps, 1)} causal pairs per step); fp64, full sort per row")
    line = {"metric": METRIC, "value": value, "unit": UNIT, "impl": "reference", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / max(args.steps, 1) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded, shapes of the workload)",
            "config": {"workload": WORKLOAD, "T": T, "S": S, "H": H, "D": D, "index_topk": TOPK},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the other workloads")
    ap.add_argument("--only", choices=sorted(OTHER_WORKLOADS),
                    help="time one of the other workloads alone (--steps calls) and print its line; "
                         "for profiling it in isolation")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    rank = _env_int("RANK", 0)
    world = _env_int("WORLD_SIZE", 1)
    local_rank = _env_int("LOCAL_RANK", 0)

    if args.impl == "reference":
        if rank == 0:
            run_reference(args)
        return

    import __graft_entry__ as g
    if rank == 0:
        g.build()
    if args.only:
        if rank == 0:
            peaks, _ = measured_peaks()
            if args.only == "chunked_prefill_fp8":
                peaks = dict(peaks)
                peaks["e4m3_tflops"] = measure_tensor_peaks(torch.device("cuda", local_rank)).get("e4m3_tflops")
            out = OTHER_WORKLOADS[args.only](torch.device("cuda", local_rank), torch.cuda.current_stream(), peaks,
                                             iters=args.steps)
            print(json.dumps({"only": args.only, **out}), flush=True)
        return
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
        torch.distributed.barrier()
        g.build()

    r = run_ours(args, rank, world, local_rank)
    if rank == 0:
        peaks, peak_kind = measured_peaks()
        score_s = r["score_ms"] / 1e3
        achieved = FLOPS / score_s / 1e12
        peak = float(peaks["bf16_tflops"])
        ms = r["total_ms"] / args.steps
        value = job_rate(PAIRS, world, ms)
        traffic = recorded_traffic()
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) q/k, N(0,1)/8 w)",
            "config": {"workload": WORKLOAD, "T": T, "S": S, "H": H, "D": D, "index_topk": TOPK,
                       "parallelism": f"replicas x{world} (independent sequences)",
                       "l2": "no flush: each step reads q (134 MB) and writes + reads 134 MB of scores, > 129 MB L2"},
            "topk_rows_per_s": job_rate(T, world, ms),
            "tc_frac_step": (FLOPS / (ms / 1e3) / 1e12) / peak,
            "kernel_ms": {"score": r["score_ms"], "topk": r["topk_ms"]},
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "kernel": "score_kernel<64,false> (tcgen05 q.k + fused ReLU/head-sum epilogue)",
                         "peak_kind": f"{peak_kind} bf16 dense burst"},
            "e2e": {"value": job_rate(PAIRS, world, r["e2e_ms"]), "unit": UNIT,
                    "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"], "steps": r["e2e_steps"]},
            "gpu_launches": 2 * args.steps,
            "clocks": r["clocks"],
            "device_status": r["status"],
        }
        if not args.no_extra:
            dev = torch.device("cuda", local_rank)
            tp = measure_tensor_peaks(dev)
            line["tensor_peaks_this_run"] = tp
            wl_peaks = dict(peaks)
            if tp.get("e4m3_tflops"):
                wl_peaks["e4m3_tflops"] = tp["e4m3_tflops"]
            line["workloads"] = run_other_workloads(dev, torch.cuda.current_stream(), wl_peaks)
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(r["case"])
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
