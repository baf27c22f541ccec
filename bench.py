"""Benchmark of one CSA2 attention layer (DeepSeek-V4.1-Flash) at decode on GB300.

Metric: CSA2 decode layer-steps/s at 128K context (Full mode: pack the new entry of every
request, score all 131,072 cached entries per request with the FP4 lightning indexer,
select the top-512, attend over them plus a 128-row bf16 window with 64 heads), and the
achieved HBM GB/s of the dominant kernel against the measured copy bandwidth.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One JSON line is printed by rank 0.  Under torchrun each rank runs its own batch of
requests (weak scaling; decode requests are independent, so there is no collective on
the data path); the timed region is bracketed by a barrier and a device synchronise and
the slowest rank's time is reported.
"""
from __future__ import annotations

import argparse
import hashlib
import concurrent.futures as cf
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "CSA2 decode layer-steps/s at 128K ctx; achieved HBM GB/s vs 8 TB/s"
UNIT = "layer-steps/s"
HEADS, HEADS_I, D, DI, TOPK, WIN = 64, 64, 512, 128, 512, 128
NOMINAL_HBM_GBS = 8000.0


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--batch", type=int, default=64, help="requests per GPU (the workload uses 64)")
    p.add_argument("--ctx", type=int, default=131072, help="cached entries per request (the workload uses 131072)")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--soak", type=float, default=1.5, help="seconds of untimed load before timing (clock sampling)")
    p.add_argument("--no-extra", action="store_true", help="skip the other workloads (tiny, Reuse/Reindex, 1M, prefill)")
    p.add_argument("--only-prefill", default=None, metavar="N0,N,G",
                   help="run only a chunked-prefill step of N new tokens on N0 cached entries, index groups of G "
                        "(--steps / --warmup iterations), print its line and exit (profiling)")
    return p.parse_args()


def workload_name(B, T):
    return f"Full-mode decode, batch {B} requests x 1 query, T={T} cached entries (ratio-1 decoder cache), " \
           f"top-512, window 128, 64 attention heads, 64 indexer heads"


# ----------------------------------------------------------------------------- distributed
def dist_init():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [x.strip() for x in vis.split(",") if x.strip()]
        self.gpu = ids[gpu_index] if gpu_index < len(ids) else str(gpu_index)
        self.proc = None
        self.lines = []
        self.t = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu), "-lms", "200"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- workload
def rank_seed_base(rank: int) -> int:
    """Seed base of a rank's replica batch: per-request seed = 1000*config + request, plus
    100,000 per rank (latent seeds base + r, key seeds base + r + 50,000, step inputs
    base + 7,000,000 + i), so the ranks' requests never share a seed."""
    return 1000 * 1 + 100000 * rank


class Workload:
    """Seeded synthetic Full-mode decode step resident on the device."""

    def __init__(self, B: int, T: int, rank: int, device):
        import synth
        from fp4_compressed_sparse_csa2_gb300 import csa2
        self.csa2 = csa2
        self.B, self.T, self.dev = B, T, device
        self.max_pages = (T + 127) // 128
        n_pages = B * self.max_pages
        self.kv = torch.empty(n_pages * csa2.KV_PAGE_BYTES, dtype=torch.uint8, device=device)
        self.idx = torch.empty(n_pages * csa2.IDX_PAGE_BYTES, dtype=torch.uint8, device=device)
        self.cache = csa2.make_cache(self.kv, self.idx, self.max_pages)
        ws0 = csa2.alloc_workspace(1, 64, 0, False, device)
        base = rank_seed_base(rank)
        self.base = base
        pos = torch.arange(T - 1, dtype=torch.int64, device=device)
        for r in range(B):
            lat = synth.torch_normal_bf16(base + r, (T - 1, D), device)
            key = synth.torch_normal_bf16(base + r + 50000, (T - 1, DI), device)
            req = torch.full((T - 1,), r, dtype=torch.int32, device=device)
            csa2.pack_kv(lat, key, req, pos, self.cache, ws0)
            del lat, key
        sb = base + 7_000_000
        self.q = synth.torch_normal_bf16(sb + 1, (B, HEADS, D), device)
        self.q_idx = synth.torch_normal_bf16(sb + 2, (B, HEADS_I, DI), device)
        self.w = synth.torch_normal_f32(sb + 3, (B, HEADS_I), device)
        self.new_lat = synth.torch_normal_bf16(sb + 4, (B, D), device)
        self.new_key = synth.torch_normal_bf16(sb + 5, (B, DI), device)
        self.window = synth.torch_normal_bf16(sb + 6, (B * WIN, D), device)
        self.req = torch.arange(B, dtype=torch.int32, device=device)
        self.nvis = torch.full((B,), T, dtype=torch.int32, device=device)
        self.win_start = torch.arange(B, dtype=torch.int64, device=device) * WIN
        self.win_len = torch.full((B,), WIN, dtype=torch.int32, device=device)
        self.new_req = torch.arange(B, dtype=torch.int32, device=device)
        self.new_pos = torch.full((B,), T - 1, dtype=torch.int64, device=device)
        self.topk_idx = torch.empty((B, TOPK), dtype=torch.int32, device=device)
        self.out = torch.empty((B, HEADS, D), dtype=torch.bfloat16, device=device)
        self.lse = torch.empty((B, HEADS), dtype=torch.float32, device=device)
        self.ws = csa2.alloc_workspace(B, HEADS_I, T, True, device)
        self.step = self.make_step(self.q, self.q_idx, self.w, self.new_lat, self.new_key, self.out)
        torch.cuda.synchronize()

    def make_step(self, q, q_idx, w, new_lat, new_key, out):
        return self.csa2.make_step(
            n_q=self.B, t_max=self.T, q=q, req=self.req, n_visible=self.nvis, window=self.window,
            win_start=self.win_start, win_len=self.win_len, cache=self.cache, topk_idx=self.topk_idx, out=out,
            lse=self.lse, q_idx=q_idx, w=w, heads_I=HEADS_I, group=1, n_new=self.B, new_latent=new_lat,
            new_idx_key=new_key, new_req=self.new_req, new_pos=self.new_pos)

    def run(self, step=None):
        self.csa2.sparse_attn_full(step or self.step, self.ws)

    # bytes the step must read from HBM (indexer keys, selected entries, window rows)
    def must_read_bytes(self):
        return self.B * (self.T * 72 + TOPK * 288 + WIN * D * 2)


# ----------------------------------------------------------------------------- oracle sample
class StepInputs:
    """The seeded inputs of one Full-mode decode step (the Workload's own draws), made with
    torch alone: the reference arm needs no CUDA library of this package."""

    def __init__(self, B: int, T: int, rank: int, device):
        import synth
        self.B, self.T, self.dev = B, T, device
        self.max_pages = (T + 127) // 128
        self.base = rank_seed_base(rank)
        sb = self.base + 7_000_000
        self.q = synth.torch_normal_bf16(sb + 1, (B, HEADS, D), device)
        self.q_idx = synth.torch_normal_bf16(sb + 2, (B, HEADS_I, DI), device)
        self.w = synth.torch_normal_f32(sb + 3, (B, HEADS_I), device)
        self.new_lat = synth.torch_normal_bf16(sb + 4, (B, D), device)
        self.new_key = synth.torch_normal_bf16(sb + 5, (B, DI), device)
        self.window = synth.torch_normal_bf16(sb + 6, (B * WIN, D), device)


def oracle_caches(wl, reqs, threads: int):
    """The resident caches of the listed requests packed by the oracle, from the same seeded
    draws as the GPU's (regenerated on the device and copied to the host one request at a
    time); built outside any timed region."""
    import oracle as orc
    import synth
    T = wl.T
    bits = lambda t: t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    caches = {}

    def build(r, lat, key):
        kv, ix = orc.alloc_pages(wl.max_pages)
        orc.pack_kv(lat, key, np.zeros(T - 1, np.int32), np.arange(T - 1, dtype=np.int64), kv, ix, None,
                    wl.max_pages)
        caches[r] = (kv, ix)

    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        futs = []
        for r in reqs:
            lat = bits(synth.torch_normal_bf16(wl.base + r, (T - 1, D), wl.dev))
            key = bits(synth.torch_normal_bf16(wl.base + r + 50000, (T - 1, DI), wl.dev))
            futs.append(ex.submit(build, r, lat, key))
            if len(futs) >= threads:        # bounds the host copies in flight
                futs.pop(0).result()
        for f in futs:
            f.result()
    return caches


def oracle_step(wl, caches, threads: int):
    """Time the CPU oracle on the Full-mode step of the requests in `caches` (pack of the new
    entry, fp64 index scores over all T entries, top-512, fp64 attention); returns seconds."""
    import oracle as orc
    T = wl.T
    bits = lambda t: t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    q, q_idx, w = bits(wl.q), bits(wl.q_idx), wl.w.cpu().numpy()
    new_lat, new_key, window = bits(wl.new_lat), bits(wl.new_key), bits(wl.window)

    def one(r):
        kv, ix = caches[r]
        orc.pack_kv(new_lat[r:r + 1], new_key[r:r + 1], np.zeros(1, np.int32), np.array([T - 1], np.int64), kv, ix,
                    None, wl.max_pages)
        I, _ = orc.index_score(q_idx[r], w[r], ix, 0, 0, T, None, wl.max_pages)
        sel = orc.topk(I.astype(np.float32), TOPK)
        orc.attention(q[r], sel, kv, 0, window[WIN * r:WIN * (r + 1)], WIN, None, None, wl.max_pages)
        return sel

    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(one, sorted(caches)))
    return time.perf_counter() - t0


def profiled_traffic(summary: str, sources, entries: int):
    """DRAM bytes per launch from a committed ncu summary under profiles/, scaled by entries scored;
    None when the kernel's sources no longer hash to the captured ones."""
    try:
        text = open(os.path.join(ROOT, "profiles", summary)).read()
    except OSError:
        return None
    m = hashlib.sha256()
    for f in sources:
        m.update(open(os.path.join(ROOT, "fp4_compressed_sparse_csa2_gb300", "csrc", f), "rb").read())
    fields = dict(re.findall(r"^(source_sha256|captured_entries): (\S+)", text, re.M))
    rd = re.search(r"dram__bytes_read\.sum \| ([0-9.]+) MB", text)
    wr = re.search(r"dram__bytes_write\.sum \| ([0-9.]+) MB", text)
    if fields.get("source_sha256") != m.hexdigest() or not rd or not wr:
        return None
    per_entry = (float(rd.group(1)) + float(wr.group(1))) * 1e6 / int(fields["captured_entries"])
    return int(round(per_entry * entries))



# ----------------------------------------------------------------------------- other workloads
def _device_cache(csa2, dev, n_req, n_entries, max_pages, seed, frac=0.0, mx=False):
    """A paged cache of n_req requests x n_entries seeded entries, packed by the library
    (mx: MXFP4 68-byte indexer keys)."""
    import synth
    n_pages = n_req * max_pages
    kv = torch.empty(n_pages * csa2.KV_PAGE_BYTES, dtype=torch.uint8, device=dev)
    idx = torch.empty(n_pages * (csa2.IDX_MX_PAGE_BYTES if mx else csa2.IDX_PAGE_BYTES), dtype=torch.uint8,
                      device=dev)
    cache = csa2.make_cache(kv, idx, max_pages, idx_format=csa2.IDX_MXFP4 if mx else csa2.IDX_E4M3_16)
    ws0 = csa2.alloc_workspace(1, 64, 0, False, dev)
    pos = torch.arange(n_entries, dtype=torch.int64, device=dev)
    for r in range(n_req):
        lat = synth.torch_normal_bf16_rows_with_outliers(seed + r, n_entries, D, frac, 8.0, dev)
        key = synth.torch_normal_bf16_rows_with_outliers(seed + r + 50000, n_entries, DI, frac, 8.0, dev)
        csa2.pack_kv(lat, key, torch.full((n_entries,), r, dtype=torch.int32, device=dev), pos, cache, ws0)
        del lat, key
    torch.cuda.synchronize()
    return cache


def _timed(csa2, fn, warmup, steps):
    """ms per call with CUDA events on the launching stream, then per-kernel device times
    from a second, traced pass."""
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    csa2.trace_enable(True)
    for _ in range(steps):
        fn()
    torch.cuda.synchronize()
    kernels = {}
    for k in csa2.TRACE_KINDS:
        tot, n = csa2.trace_read(k)
        if n:
            kernels[k] = round(1000 * tot / n, 2)
    csa2.trace_enable(False)
    return ms, kernels


def _decode_line(csa2, dev, name, B, T, seed, frac=0.0, steps=10, warmup=3, sinks_rope=False, ring=False, mx=False):
    import synth
    mp = (T + 127) // 128
    cache = _device_cache(csa2, dev, B, T - 1, mp, seed, frac, mx)
    sb = seed + 7_000_000
    q = synth.torch_normal_bf16(sb + 1, (B, HEADS, D), dev)
    q_idx = synth.torch_normal_bf16(sb + 2, (B, HEADS_I, DI), dev)
    w = synth.torch_normal_f32(sb + 3, (B, HEADS_I), dev)
    new_lat = synth.torch_normal_bf16(sb + 4, (B, D), dev)
    new_key = synth.torch_normal_bf16(sb + 5, (B, DI), dev)
    window = synth.torch_normal_bf16(sb + 6, (B * WIN, D), dev)
    out = torch.empty((B, HEADS, D), dtype=torch.bfloat16, device=dev)
    extra = {}
    if sinks_rope:  # per-head sinks and the partial RoPE of q and O, angles of position T - 1
        ang = (T - 1) * torch.pow(10000.0, -torch.arange(32, dtype=torch.float64, device=dev) / 32.0)
        extra = {"sinks": synth.torch_normal_f32(sb + 7, (HEADS,), dev),
                 "rope_cos": torch.cos(ang).float().expand(B, 32).contiguous(),
                 "rope_sin": torch.sin(ang).float().expand(B, 32).contiguous()}
    kw = dict(n_q=B, t_max=T, q=q, req=torch.arange(B, dtype=torch.int32, device=dev),
              n_visible=torch.full((B,), T, dtype=torch.int32, device=dev), window=window,
              win_start=torch.arange(B, dtype=torch.int64, device=dev) * WIN,
              win_len=torch.full((B,), WIN, dtype=torch.int32, device=dev), cache=cache,
              topk_idx=torch.empty((B, TOPK), dtype=torch.int32, device=dev), out=out,
              lse=torch.empty((B, HEADS), dtype=torch.float32, device=dev), q_idx=q_idx, w=w,
              heads_I=HEADS_I, group=1, n_new=B, new_latent=new_lat, new_idx_key=new_key,
              new_req=torch.arange(B, dtype=torch.int32, device=dev),
              new_pos=torch.full((B,), T - 1, dtype=torch.int64, device=dev), **extra)
    step = csa2.make_step(**kw)
    ws = csa2.alloc_workspace(B, HEADS_I, T, True, dev)
    run = lambda: csa2.sparse_attn_full(step, ws)
    if ring:  # FP8 window ring: the 127 earlier window entries packed once, the step's own each step
        wring = torch.zeros(B * WIN * 528, dtype=torch.uint8, device=dev)
        req = torch.arange(B, dtype=torch.int32, device=dev)
        for j in range(WIN - 1):
            csa2.pack_window(window[j::WIN].contiguous(), req, torch.full((B,), T - WIN + j, dtype=torch.int64,
                                                                             device=dev), wring, B, ws)
        own = window[WIN - 1::WIN].contiguous()
        own_pos = torch.full((B,), T - 1, dtype=torch.int64, device=dev)
        step = csa2.make_step(**{**kw, "window": None, "win_ring": wring, "win_ring_reqs": B, "win_start": own_pos})

        def run():
            csa2.pack_window(own, req, own_pos, wring, B, ws)
            csa2.sparse_attn_full(step, ws)
    ms, kernels = _timed(csa2, run, warmup, steps)
    st, info = csa2.check(ws)
    key_bytes = 68 if mx else 72
    must = B * (T * key_bytes + TOPK * 288 + WIN * (528 if ring else D * 2))
    return {"workload": name, "metric": UNIT, "value": round(1000.0 / ms, 2), "ms_per_step": round(ms, 4),
            "must_read_bytes": must, "step_gbs": round(must / (ms * 1e-3) / 1e9, 1),
            "index_gbs": round(B * T * key_bytes / (kernels.get("index", float("nan")) * 1e-6) / 1e9, 1),
            "kernels_us": kernels, "device_status": st}


def mma_peaks(dev):
    """Tensor-core rates of this library's instruction shapes, measured with the probe
    kernel (csa2_probe_mma): every SM issues 8,192 MMAs per issuer back to back; TFLOP/s from
    CUDA events around the launch, MAC per cycle per SM from the kernel's own clock."""
    from fp4_compressed_sparse_csa2_gb300 import csa2
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    cyc = torch.zeros(sms, dtype=torch.int64, device=dev)
    out = {}
    for kind, name, K, shapes in [(1, "nvf4", 64, [(64, 4), (128, 2), (128, 3), (256, 1)]),
                                  (0, "f16", 16, [(64, 4), (128, 2), (256, 1)])]:
        for n, iss in shapes:
            iters = 8192
            csa2.probe_mma(kind, n, 64, iss, sms, cyc)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            csa2.probe_mma(kind, n, iters, iss, sms, cyc)
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1)
            macs = 128 * n * K * iters * iss
            out[f"{name}_n{n}_i{iss}"] = {"tflops": round(2 * macs * sms / (ms * 1e-3) / 1e12, 1),
                                          "mac_per_cycle_sm": round(macs / float(cyc.float().median()), 0)}
    out["nvf4_peak_tflops"] = max(v["tflops"] for k, v in out.items() if k.startswith("nvf4"))
    out["f16_peak_tflops"] = max(v["tflops"] for k, v in out.items() if k.startswith("f16_"))
    return out


PREFILL_GROUP = 1  # queries per indexer MMA group in the chunked-prefill line


def prefill_line(dev, n0, n, group, warmup=2, steps=5, probe=True):
    """A chunked-prefill step: n new tokens appended causally to n0 cached entries of one
    request (pack the new entries, causally masked index scores in groups of `group`
    queries, top-512 per query, attention over the selection and each query's 128-row
    window), with the indexer's FP4 rate against the probe-measured peak."""
    import synth
    from fp4_compressed_sparse_csa2_gb300 import csa2
    T = n0 + n
    mp = (T + 127) // 128
    cache = _device_cache(csa2, dev, 1, n0, mp, 4000)
    sb = 4000 + 7_000_000
    new_lat = synth.torch_normal_bf16(sb + 4, (n, D), dev)
    new_key = synth.torch_normal_bf16(sb + 5, (n, DI), dev)
    rows = torch.cat([synth.torch_normal_bf16(sb + 6, (127, D), dev), new_lat]).contiguous()
    step = csa2.make_step(n_q=n, t_max=T, q=synth.torch_normal_bf16(sb + 1, (n, HEADS, D), dev),
                          req=torch.zeros(n, dtype=torch.int32, device=dev),
                          n_visible=torch.arange(n0 + 1, T + 1, dtype=torch.int32, device=dev), window=rows,
                          win_start=torch.arange(n, dtype=torch.int64, device=dev),
                          win_len=torch.full((n,), WIN, dtype=torch.int32, device=dev), cache=cache,
                          topk_idx=torch.empty((n, TOPK), dtype=torch.int32, device=dev),
                          out=torch.empty((n, HEADS, D), dtype=torch.bfloat16, device=dev),
                          lse=torch.empty((n, HEADS), dtype=torch.float32, device=dev),
                          q_idx=synth.torch_normal_bf16(sb + 2, (n, HEADS_I, DI), dev),
                          w=synth.torch_normal_f32(sb + 3, (n, HEADS_I), dev), heads_I=HEADS_I, group=group,
                          n_new=n, new_latent=new_lat, new_idx_key=new_key,
                          new_req=torch.zeros(n, dtype=torch.int32, device=dev),
                          new_pos=torch.arange(n0, T, dtype=torch.int64, device=dev))
    ws = csa2.alloc_workspace(n, HEADS_I, T, True, dev)
    ms, kernels = _timed(csa2, lambda: csa2.sparse_attn_full(step, ws), warmup, steps)
    st, _ = csa2.check(ws)
    pairs = n * n0 + n * (n + 1) // 2                 # visible (query, entry) pairs
    flops = pairs * HEADS_I * DI * 2
    del step, ws, cache
    torch.cuda.empty_cache()
    line = {"workload": f"chunked prefill: {n} new tokens on {n0} cached entries, index groups of {group}",
            "metric": "chunk-steps/s", "value": round(1000.0 / ms, 3), "ms_per_step": round(ms, 3),
            "kernels_us": kernels, "index_flops": flops, "device_status": st}
    idx_tf = flops / (kernels.get("index", float("nan")) * 1e-6) / 1e12
    line["index_tflops"] = round(idx_tf, 1)
    if probe:
        pk = mma_peaks(dev)
        line.update({"index_fp4_frac": round(idx_tf / pk["nvf4_peak_tflops"], 4),
                     "fp4_peak_tflops": round(pk["nvf4_peak_tflops"], 1),
                     "fp4_peak_source": "measured: csa2_probe_mma, back-to-back block-scaled NVFP4 tcgen05.mma "
                                        "(M=128, best of N and issuer counts) on every SM, CUDA events",
                     "mma_probe": pk})
    return line


def measure_extra(dev, hbm_peak, bf16_tflops):
    """The other workloads of the layer, each in its own line: the tiny decode, Reuse and
    Reindex at 128 x 262,144, the headline decode with sinks and fused partial RoPE, with the
    FP8 window ring and with MXFP4 indexer keys, the
    million-token decode with its ratio-2 layer (1 % of entries x 8), and a 4,096-token
    chunked prefill on 262,144 cached entries."""
    import synth
    from fp4_compressed_sparse_csa2_gb300 import csa2
    lines = []

    def attempt(fn):
        try:
            lines.append(fn())
        except Exception as exc:  # a failed extra workload is reported, the headline stands
            lines.append({"error": f"{type(exc).__name__}: {exc}"[:300]})
        torch.cuda.synchronize()
        torch.cuda.empty_cache()

    attempt(lambda: dict(_decode_line(csa2, dev, "tiny Full decode, B=1, T=4096 (L2-resident)", 1, 4096, 0),
                         note="launch-latency bound"))

    def reuse_reindex():
        B, T = 128, 262144
        mp = T // 128
        cache = _device_cache(csa2, dev, B, T, mp, 2000)
        q = synth.torch_normal_bf16(2000 + 7_000_001, (B, HEADS, D), dev)
        window = synth.torch_normal_bf16(2000 + 7_000_006, (B * WIN, D), dev)
        common = dict(n_q=B, t_max=T, q=q, req=torch.arange(B, dtype=torch.int32, device=dev),
                      n_visible=torch.full((B,), T, dtype=torch.int32, device=dev), window=window,
                      win_start=torch.arange(B, dtype=torch.int64, device=dev) * WIN,
                      win_len=torch.full((B,), WIN, dtype=torch.int32, device=dev), cache=cache,
                      out=torch.empty((B, HEADS, D), dtype=torch.bfloat16, device=dev),
                      lse=torch.empty((B, HEADS), dtype=torch.float32, device=dev))
        sel = synth.torch_distinct_indices(2000 + 7_000_007, B, T, TOPK, dev)
        ws = csa2.alloc_workspace(B, HEADS_I, T, True, dev)
        reuse = csa2.make_step(topk_idx=sel, **common)
        ms_u, k_u = _timed(csa2, lambda: csa2.sparse_attn_reuse(reuse, ws), 3, 20)
        reidx = csa2.make_step(topk_idx=torch.empty((B, TOPK), dtype=torch.int32, device=dev),
                               q_idx=synth.torch_normal_bf16(2000 + 7_000_002, (B, HEADS_I, DI), dev),
                               w=synth.torch_normal_f32(2000 + 7_000_003, (B, HEADS_I), dev), heads_I=HEADS_I,
                               **common)
        ms_r, k_r = _timed(csa2, lambda: csa2.sparse_attn_reindex(reidx, ws), 3, 10)
        st, _ = csa2.check(ws)
        must_u = B * (TOPK * 288 + WIN * D * 2)
        must_r = B * (T * 72) + must_u
        return {"workload": "Reuse and Reindex decode, B=128, T=262144", "metric": UNIT,
                "reuse": {"value": round(1000.0 / ms_u, 2), "ms_per_step": round(ms_u, 4), "kernels_us": k_u,
                          "must_read_bytes": must_u, "step_gbs": round(must_u / (ms_u * 1e-3) / 1e9, 1)},
                "reindex": {"value": round(1000.0 / ms_r, 2), "ms_per_step": round(ms_r, 4), "kernels_us": k_r,
                            "must_read_bytes": must_r, "step_gbs": round(must_r / (ms_r * 1e-3) / 1e9, 1),
                            "index_gbs": round(B * T * 72 / (k_r.get("index", float("nan")) * 1e-6) / 1e9, 1)},
                "device_status": st}

    attempt(reuse_reindex)
    attempt(lambda: dict(_decode_line(csa2, dev, "Full decode with per-head sinks and fused partial RoPE, B=64, "
                                      "T=131072", 64, 131072, 3200, sinks_rope=True), note="next row N4"))
    attempt(lambda: dict(_decode_line(csa2, dev, "Full decode with the FP8 window ring (the step's own window entry "
                                      "packed each step), B=64, T=131072", 64, 131072, 3300, ring=True),
                         note="next row N2"))
    attempt(lambda: dict(_decode_line(csa2, dev, "Full decode with MXFP4 68-byte indexer keys (E8M0 per 32 "
                                      "channels), B=64, T=131072", 64, 131072, 3400, mx=True), note="next row N3"))
    def hierarchical():
        # a Full layer that also publishes its candidate pool, then a Reindex layer that
        # scores only the pool (16,384 positions) with its own query
        B, T = 64, 131072
        mp = T // 128
        cache = _device_cache(csa2, dev, B, T, mp, 3500)
        sb = 3500 + 7_000_000
        common = dict(n_q=B, t_max=T, q=synth.torch_normal_bf16(sb + 1, (B, HEADS, D), dev),
                      req=torch.arange(B, dtype=torch.int32, device=dev),
                      n_visible=torch.full((B,), T, dtype=torch.int32, device=dev),
                      window=synth.torch_normal_bf16(sb + 6, (B * WIN, D), dev),
                      win_start=torch.arange(B, dtype=torch.int64, device=dev) * WIN,
                      win_len=torch.full((B,), WIN, dtype=torch.int32, device=dev), cache=cache,
                      topk_idx=torch.empty((B, TOPK), dtype=torch.int32, device=dev),
                      out=torch.empty((B, HEADS, D), dtype=torch.bfloat16, device=dev),
                      lse=torch.empty((B, HEADS), dtype=torch.float32, device=dev), heads_I=HEADS_I)
        pool = torch.empty((B, csa2.POOL), dtype=torch.int32, device=dev)
        ws = csa2.alloc_workspace(B, HEADS_I, T, True, dev, pool=True)
        full = csa2.make_step(q_idx=synth.torch_normal_bf16(sb + 2, (B, HEADS_I, DI), dev),
                              w=synth.torch_normal_f32(sb + 3, (B, HEADS_I), dev), pool=pool, **common)
        ms_f, k_f = _timed(csa2, lambda: csa2.sparse_attn_full(full, ws), 3, 10)
        reidx = csa2.make_step(q_idx=synth.torch_normal_bf16(sb + 4, (B, HEADS_I, DI), dev),
                               w=synth.torch_normal_f32(sb + 5, (B, HEADS_I), dev), pool=pool, **common)
        ms_r, k_r = _timed(csa2, lambda: csa2.sparse_attn_reindex(reidx, ws), 3, 20)
        st, _ = csa2.check(ws)
        must_r = B * (csa2.POOL * 72 + TOPK * 288 + WIN * D * 2)
        return {"workload": "hierarchical indexer, B=64, T=131072: Full publishing its 16,384-position pool, "
                            "then a Reindex over the pool", "metric": UNIT,
                "full_with_pool": {"value": round(1000.0 / ms_f, 2), "ms_per_step": round(ms_f, 4),
                                   "kernels_us": k_f},
                "reindex_over_pool": {"value": round(1000.0 / ms_r, 2), "ms_per_step": round(ms_r, 4),
                                      "kernels_us": k_r, "must_read_bytes": must_r,
                                      "step_gbs": round(must_r / (ms_r * 1e-3) / 1e9, 1)},
                "device_status": st, "note": "next row N1"}

    attempt(hierarchical)
    attempt(lambda: dict(_decode_line(csa2, dev, "million-token Full decode, B=8, T=1048576, 1% of entries x8", 8,
                                      1 << 20, 3000, 0.01), note="decoder layer"))
    attempt(lambda: dict(_decode_line(csa2, dev, "ratio-2 layer Full decode, B=8, 524288 pooled entries, 1% x8", 8,
                                      1 << 19, 3100, 0.01), note="encoder-style layer of the same step"))

    attempt(lambda: prefill_line(dev, 262144, 4096, PREFILL_GROUP))
    return lines

def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ----------------------------------------------------------------------------- arms
def run_ours(args, ws, rank, local):
    dev = torch.device("cuda", local)
    from fp4_compressed_sparse_csa2_gb300 import csa2
    wl = Workload(args.batch, args.ctx, rank, dev)
    stream = torch.cuda.current_stream()
    for _ in range(max(args.warmup, 3)):
        wl.run()
    st, info = csa2.check(wl.ws)
    assert st == csa2.OK, f"device error word {st} info {info}"
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        # untimed soak so that the sampler (200 ms period) sees the GPU under this load
        t_end = time.time() + args.soak
        while time.time() < t_end:
            for _ in range(20):
                wl.run()
            torch.cuda.synchronize()
        barrier(ws)
        torch.cuda.synchronize()
        l0 = csa2.launch_count()
        ev0.record(stream)
        for _ in range(args.steps):
            wl.run()
        ev1.record(stream)
        torch.cuda.synchronize()
        launches = csa2.launch_count() - l0
    barrier(ws)
    ms = ev0.elapsed_time(ev1) / args.steps
    # per-kernel device times from a second, traced pass of the same steps (the trace puts
    # CUDA events between the kernels, so the headline above is timed without it)
    csa2.trace_enable(True)
    for _ in range(args.steps):
        wl.run()
    torch.cuda.synchronize()
    kernels = {}
    for k in csa2.TRACE_KINDS:
        tot, n = csa2.trace_read(k)
        if n:
            kernels[k] = {"us_per_launch": 1000 * tot / n, "launches": n}
    csa2.trace_enable(False)
    st, info = csa2.check(wl.ws)
    assert st == csa2.OK, f"device error word {st} info {info}"
    ms = max_over_ranks(ms, ws)
    value = ws / (ms / 1000.0)

    # roofline of the dominant kernel (the indexer): algorithmic bytes = 72 B per scored entry
    idx_us = kernels["index"]["us_per_launch"]
    idx_bytes = wl.B * wl.T * 72
    traffic = profiled_traffic("index_kernel_decode_b16_t131072.md", ("k_index.cu", "csa2_dev.cuh", "csa2_kernels.cuh"),
                               wl.B * wl.T)
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except OSError:
        pass
    hbm_peak = float(peaks.get("hbm_gbs", 6800.0))
    achieved = idx_bytes / (idx_us * 1e-6) / 1e9
    roofline = {"bound": "hbm", "kernel": "index_kernel", "achieved": round(achieved, 1),
                "peak": hbm_peak, "unit": "GB/s", "frac": round(achieved / hbm_peak, 4),
                "peak_source": "measured (MEASURED_PEAKS.json hbm_gbs)" if peaks else "fallback 6.8 TB/s",
                "traffic": traffic, "algorithmic_bytes": idx_bytes,
                "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum of a 16-request capture, scaled "
                                  "by entries scored (null once the kernel source differs from the capture's)"}
    # the same kernel inside a launch chain, as in the untraced step: csa2_index_score back
    # to back (each call packs its query first; the indexer copies its first key pages while
    # that runs), CUDA events around the calls -- context for the traced figure above, whose
    # events between the kernels break the chaining
    sc_i = torch.empty((wl.B, wl.T), dtype=torch.float32, device=dev)
    ws_i = csa2.alloc_workspace(wl.B, HEADS_I, wl.T, False, dev)
    run_i = lambda: csa2.index_score(wl.q_idx, wl.w, HEADS_I, wl.req, wl.nvis, wl.B, 1, wl.T, wl.cache, sc_i, wl.T, ws_i)
    for _ in range(3):
        run_i()
    torch.cuda.synchronize()
    ci0, ci1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ci0.record(stream)
    for _ in range(20):
        run_i()
    ci1.record(stream)
    torch.cuda.synchronize()
    ch_us = ci0.elapsed_time(ci1) / 20 * 1e3
    st_i, _ = csa2.check(ws_i)
    assert st_i == csa2.OK, f"device error word {st_i}"
    ch_gbs = idx_bytes / (ch_us * 1e-6) / 1e9
    roofline["chained"] = {"us_per_call": round(ch_us, 2), "achieved": round(ch_gbs, 1), "frac": round(ch_gbs / hbm_peak, 4),
                           "how": "csa2_index_score called 20 times back to back (query packing + indexer per call)"}
    del sc_i, ws_i
    step_gbs = wl.must_read_bytes() / (ms * 1e-3) / 1e9

    # end to end through the C ABI with host buffers: every step copies its inputs in from
    # pinned host memory and its output back; two buffer sets and separate copy streams
    # let the copies of neighbouring steps overlap a step's kernels (the kernels of
    # consecutive steps stay ordered on the compute stream: each reads the cache the
    # previous one appended to)
    e2e = None
    if not args.no_e2e:
        pin = lambda t: t.cpu().pin_memory()
        hin = [pin(x) for x in (wl.q, wl.q_idx, wl.w, wl.new_lat, wl.new_key)]
        h2d = sum(x.numel() * x.element_size() for x in hin)
        sets = []
        for _ in range(2):
            din = [torch.empty_like(x) for x in (wl.q, wl.q_idx, wl.w, wl.new_lat, wl.new_key)]
            dout = torch.empty_like(wl.out)
            hout = torch.empty(wl.out.shape, dtype=wl.out.dtype).pin_memory()
            sets.append({"din": din, "dout": dout, "hout": hout, "step": wl.make_step(*din, dout),
                         "in_done": torch.cuda.Event(), "run_done": torch.cuda.Event(),
                         "out_done": torch.cuda.Event(), "used": False})
        d2h = sets[0]["hout"].numel() * sets[0]["hout"].element_size()
        up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

        def e2e_steps(n):
            for i in range(n):
                st_ = sets[i & 1]
                with torch.cuda.stream(up):
                    if st_["used"]:  # the set's previous step has read its inputs and written its output
                        up.wait_event(st_["run_done"])
                    for d_, h_ in zip(st_["din"], hin):
                        d_.copy_(h_, non_blocking=True)
                    st_["in_done"].record(up)
                stream.wait_event(st_["in_done"])
                if st_["used"]:  # the previous output of this set is on the host before it is overwritten
                    stream.wait_event(st_["out_done"])
                wl.run(st_["step"])
                st_["run_done"].record(stream)
                with torch.cuda.stream(down):
                    down.wait_event(st_["run_done"])
                    st_["hout"].copy_(st_["dout"], non_blocking=True)
                    st_["out_done"].record(down)
                st_["used"] = True

        e2e_steps(max(args.warmup, 3))
        torch.cuda.synchronize()
        barrier(ws)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(up)  # before the first step's input copies
        e2e_steps(args.steps)
        down.wait_stream(up)
        down.wait_stream(stream)
        e1.record(down)  # after the last step's output copy
        torch.cuda.synchronize()
        barrier(ws)
        ems = max_over_ranks(e0.elapsed_time(e1) / args.steps, ws)
        e2e = {"value": round(ws / (ems / 1000.0), 2), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "ms_per_step": round(ems, 4),
               "pipelining": "inputs of step i+1 copied in and the output of step i copied out while kernels run "
                             "(two buffer sets, copy streams)"}

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu:
        cores = host_cores()
        n_req = min(wl.B, max(4, cores))
        nr = n_req
        secs = oracle_step(wl, oracle_caches(wl, list(range(n_req)), cores), cores)
        cpu = {"value": round((nr / wl.B) / secs, 6), "unit": UNIT, "cores": min(cores, nr), "kind": "oracle",
               "sample": f"{nr} of {wl.B} requests of the same Full-mode step (pack + fp64 index scores over "
                         f"{wl.T} entries + top-512 + fp64 attention), {secs:.2f} s wall on {min(cores, nr)} "
                         f"threads, scaled to one {wl.B}-request layer-step"}

    clocks = clk.summary()
    extra = None
    if rank == 0 and ws == 1 and not args.no_extra:
        extra = measure_extra(dev, hbm_peak, float(peaks.get("bf16_tflops", 1900.0)))
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": round(ms, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "fp4e2m1 x fp4e2m1 (indexer), f16 (attention), fp32 acc",
            "data": "synthetic (seeded N(0,1) latents, keys, queries; fp32 N(0,1) head weights)",
            "config": {"workload": workload_name(wl.B, wl.T), "global_batch": wl.B * ws, "seq_len": wl.T,
                       "parallelism": f"replicas x{ws} (requests sharded, no collective)",
                       "l2": f"inputs larger than L2: {wl.B * wl.T * 72 / 1e6:.0f} MB of indexer keys per step "
                             f"stream from HBM"},
            "hbm": {"must_read_bytes_per_step": wl.must_read_bytes(), "step_gbs": round(step_gbs, 1),
                    "frac_of_8tbs": round(step_gbs / NOMINAL_HBM_GBS, 4),
                    "frac_of_measured": round(step_gbs / hbm_peak, 4)},
            "roofline": roofline,
            "kernels": {k: {"us_per_launch": round(v["us_per_launch"], 2), "launches": v["launches"]}
                        for k, v in kernels.items()},
            "gpu_launches": int(launches),
            "e2e": e2e, "cpu_baseline": cpu, "clocks": clocks,
            "extra": extra,
        }
        print(json.dumps(line), flush=True)


def run_reference(args, ws, rank, local):
    """The oracle as it stands, on the host cores: whole Full-mode layer-steps (every request
    of the batch), timed one by one.  Inputs are the GPU arm's seeded draws made with torch
    alone; no CUDA library of this package is loaded."""
    if rank != 0:
        return
    dev = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
    wl = StepInputs(args.batch, args.ctx, 0, dev)
    cores = host_cores()
    caches = oracle_caches(wl, list(range(wl.B)), cores)
    warm = max(0, min(args.warmup, 1))
    for _ in range(warm):
        oracle_step(wl, {0: caches[0]}, 1)
    steps = max(1, min(args.steps, 3))
    times = [oracle_step(wl, caches, cores) for _ in range(steps)]
    sec = statistics.median(times)
    value = 1.0 / sec
    line = {
        "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": ws, "steps": steps,
        "warmup": warm, "ms_per_step": round(sec * 1000, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "impl": "reference",
        "data": "synthetic (seeded N(0,1)), same inputs as the GPU arm",
        "config": {"workload": workload_name(wl.B, wl.T), "global_batch": wl.B, "seq_len": wl.T},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": min(cores, wl.B), "kind": "oracle",
                         "sample": f"whole layer-steps: all {wl.B} requests per step, {steps} steps timed one by "
                                   f"one (median), caches packed by the oracle outside the timed region"},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.only_prefill:
        n0, n, g = (int(x) for x in args.only_prefill.split(","))
        dev = torch.device("cuda", 0)
        print(json.dumps(prefill_line(dev, n0, n, g, warmup=max(args.warmup, 1), steps=max(args.steps, 1),
                                      probe=False)), flush=True)
        return
    ws, rank, local = dist_init()
    if args.impl == "reference":
        run_reference(args, ws, rank, local)
    else:
        run_ours(args, ws, rank, local)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
