"""Benchmark: paged MLA decode latent-cache bandwidth on GB300.

One step = the hot path over one batch: write the step's new cache rows
(mla_cache_write) and decode every request against the paged latent cache
(mla_decode, which includes the split merge). Metric: latent-cache GB/s =
(sum of context tokens x row bytes) / step time, each request's rows counted
once; also decode steps/s and context tokens/s.

  python bench.py [--gpus N] [--steps K] [--warmup W]
                  [--config mtp|batched|long|fp8|tiny|verify|verify8|latent768]
                  [--side long,fp8,...|none] [--clock-csv PATH] [--requests N]
  python bench.py --impl reference ...   # the CPU oracle on the same workload
  python bench.py --config gather        # the fp8_ds_mla prefill-context gather (mla_gather_upconvert)

The headline workload (default mtp: the 9.8M-slot pool, 128 requests of up
to 100k tokens, 4-token causal verify steps, the largest configuration that
fits one GPU) gives the line's value, roofline, e2e and cpu_baseline; the
other workloads (--side) are measured the same way afterwards and reported
under "workloads" in the same line.

Timing: W untimed warm-up steps, then K steps, each bracketed by CUDA events
on the launching stream, with L2 flushed (a 256 MiB write) before every step
outside the events; barrier + synchronize around the timed region; the max
over ranks is reported. Under torchrun every rank runs an independent replica
(its own seeded batch): requests are independent, so there is no collective
on the data path and scaling is weak.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MLA paged decode latent-cache HBM GB/s (% of GB300 peak) and decode steps/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
DECODE_SRC = os.path.join(ROOT, "mla_latent_kv_cache_gb300", "csrc", "decode.cu")
GATHER_SRC = os.path.join(ROOT, "mla_latent_kv_cache_gb300", "csrc", "cache_write.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
CONFIG_TEXT = {
    "tiny": "B=2 Hq=8 seq {37,200} page 16 bf16",
    "batched": "B=64 Hq=16 seq U{1024..8192} page 16 bf16",
    "long": "B=4 Hq=32 seq 262144 page 64 bf16",
    "mtp": "B=128 Hq=16 Qt=4 causal, 9.8M-slot pool above slot 3,728,270, seq 0/1/U{2048..100000}, page 16 bf16",
    "fp8": "B=64 Hq=64 seq 32768 page 64 fp8_ds_mla (656 B rows)",
    "verify": "the mtp workload with a verify length of its own per request, U{1..4} (seeded): "
              "mla_decode_varlen",
    "verify8": "the mtp pool and requests with verify steps of 1 + k tokens, k U{0..7} per request (seeded; up "
               "to 128 query rows a request, one cache read each): mla_decode_varlen",
    "latent768": "the batched shape (B=64 Hq=16 seq U{1024..8192} page 16) over bf16 rows [latent 768 | rope 64] "
                 "(1664 B): mla_cache_write_latent + mla_decode_latent",
    "gather": "fp8_ds_mla pool of the fp8 workload (B=64 x 32768 tokens, page 64) gathered into "
              "[2097152, 576] bf16 rows",
}
GATHER_METRIC = "fp8_ds_mla context gather + upconvert HBM GB/s (656 B read + 1152 B written per token)"
GATHER_BYTES_PER_TOKEN = 656 + 1152


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_over_ranks(values, op):
    """values: list of floats on this rank -> reduced over ranks ("max"/"sum")."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return list(values)
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor(values, dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return t.cpu().tolist()


def aggregate(bytes_per_step, ms_per_step):
    """Whole-job throughput: bytes of all ranks / the slowest rank's time."""
    tot_bytes = reduce_over_ranks([bytes_per_step], "sum")[0]
    ms = reduce_over_ranks([ms_per_step], "max")[0]
    return tot_bytes, ms


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


KERNEL_HEADERS = [os.path.join(ROOT, "mla_latent_kv_cache_gb300", "csrc", f)
                  for f in ("launch.cuh", "mla_common.cuh", "tmem_ldst.inc")]


def _code_only(text):
    """C/C++ source with comments and blank space removed (string and
    character literals kept), so that a comment edit keeps a capture valid."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            i = text.find("\n", i)
            i = n if i < 0 else i
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_sha(src=DECODE_SRC):
    """Hash of the code (comments stripped) of a kernel file and the headers
    it includes: a committed ncu traffic figure holds only while it matches."""
    h = hashlib.sha256()
    for f in [src] + KERNEL_HEADERS:
        h.update(_code_only(open(f, encoding="utf-8").read()).encode())
    return h.hexdigest()[:16]


def traffic_for(config):
    """DRAM bytes per launch of the workload's dominant kernel from a committed
    ncu capture, if it was taken on the current kernel source; else None."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    d = json.load(open(TRAFFIC_FILE))
    e = d.get(config)
    if not e or e.get("kernel_src_sha") != kernel_sha(GATHER_SRC if config == "gather" else DECODE_SRC):
        return None
    return e.get("dram_bytes_per_launch")


def timing_events(n, stream):
    """n pairs of timing events, each recorded once so that the CUDA events
    exist before the timed loop (torch creates an event on its first record):
    the loop then makes no event-creating driver calls."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for a, b in evs:
        a.record(stream)
        b.record(stream)
    return evs


def step_time_summary(times_ms):
    """Median step time and the steps that took over ten times it (and over a
    millisecond): a stall of the device or the host inside a step's events
    shows up here rather than only as a lower mean."""
    t = sorted(times_ms)
    med = t[len(t) // 2]
    slow = [x for x in times_ms if x > 10 * med and x > 1.0]
    return {"median_ms": round(med, 5), "stalled_steps": len(slow), "stalled_ms": round(sum(slow) - med * len(slow), 1)}


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    # Three fields per sample: the throttle reasons come from the one bitmask
    # (NVML's clocks-event-reason bits), not five separate queries, and there
    # is no power reading. With nine fields (power and each reason on its
    # own) polled every 50 or 200 ms, a timed region of about a second now and
    # then took whole seconds longer, the time landing inside the steps' events
    # (and the JSON line's stalled_steps saying so).
    Q = "index,clocks.sm,clocks.max.sm,clocks_event_reasons.active"
    REASON_BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
                   "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80}

    def __init__(self, gpu_index: int, out_path: str | None):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.out_path = out_path
        self.first_timed = 0  # index of the first sample taken inside the timed region

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (FileNotFoundError, OSError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def mark(self):
        """The timed region starts: clock statistics use the samples from here on."""
        self.first_timed = len(self.lines)

    def wait_first(self, settle_s: float = 1.0, samples: int = 3, timeout_s: float = 10.0):
        """Block until nvidia-smi has run for `settle_s` and produced `samples`
        samples, so its start-up is over before the warm-up and timing."""
        t0 = time.perf_counter()
        while self.proc is not None and time.perf_counter() - t0 < timeout_s:
            if len(self.lines) >= samples and time.perf_counter() - t0 >= settle_s:
                break
            time.sleep(0.05)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        if self.out_path:
            with open(self.out_path, "w") as f:
                f.write(self.Q + "\n" + "\n".join(self.lines) + "\n")
        return self.summarize(self.lines[self.first_timed:] or self.lines)

    @classmethod
    def summarize(cls, lines):
        """Median SM clock, the maximum clock and the throttle reasons seen in
        nvidia-smi csv lines of the fields in Q."""
        sm, mx, reasons = [], [], set()
        for ln in lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 4:
                continue
            try:
                clk, clk_max, bits = float(parts[1]), float(parts[2]), int(parts[3], 16)
            except ValueError:
                continue
            sm.append(clk)
            mx.append(clk_max)
            reasons.update(n for n, bit in cls.REASON_BITS.items() if bits & bit)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- GPU arm

def verify_qlens(B, rank=0, qmax=4):
    """The verify workloads' per-request verify lengths, U{1..qmax} (seeded)."""
    import numpy as np
    return np.random.default_rng(7 + 1000 * rank).integers(1, qmax + 1, size=B)


WORKLOAD_SEED = {"tiny": 1, "batched": 2, "long": 3, "mtp": 4, "fp8": 5}
# workloads measured beside the headline one and reported in its line
SIDE_WORKLOADS = ("long", "fp8", "batched", "tiny", "verify", "verify8", "latent768")


def config_dict(name, ctx_tokens, cache_bytes, row_bytes, ws_):
    """The `config` object of a decode line; both arms use it, so the
    reference arm's line names the same workload in the same words."""
    varlen = name.startswith("verify")
    lat = name.startswith("latent")
    return {"workload": name, "shape": CONFIG_TEXT[name], "context_tokens": ctx_tokens,
            "cache_bytes_per_step": cache_bytes, "row_bytes": row_bytes,
            "l2": "flushed before every step (256 MiB write, outside the timed events)",
            "step": ("mla_cache_write_latent" if lat else "mla_cache_write") + " of the step's new rows + "
                    + ("mla_decode_varlen" if varlen else "mla_decode_latent" if lat else "mla_decode")
                    + " (decode + split merge)",
            "parallelism": f"replicas x{ws_} (requests are independent)"}


def build_workload(name, dev, rank=0, requests=None):
    """The named workload on `dev` (verify: the mtp workload's pool and
    requests), seeded per rank. `requests` (long, fp8 and mtp only) keeps
    that many of their requests: a cut-down copy for profiling."""
    from mla_latent_kv_cache_gb300 import workloads as W
    if name.startswith("latent"):
        return W.latent(int(name[len("latent"):]), device=dev, seed=WORKLOAD_SEED["batched"] + 1000 * rank)
    base = "mtp" if name.startswith("verify") else name
    kw = {"Qt": 8} if name == "verify8" else {}
    if requests is not None:
        if name not in ("long", "fp8", "mtp"):
            raise SystemExit("--requests applies to the long, fp8 and mtp workloads only")
        kw["B"] = int(requests)
    return W.CONFIGS[base](device=dev, seed=WORKLOAD_SEED[base] + 1000 * rank, **kw)


def measure_gpu(name, args, dev, rank, ws_, clock_csv=None):
    """Time K steps of workload `name` (device-resident inputs), then the
    same step end to end from pinned host memory. Returns the numbers of one
    JSON line (before the max over ranks)."""
    import numpy as np
    import torch
    import torch.distributed as dist
    import mla_latent_kv_cache_gb300 as m

    varlen = name.startswith("verify")
    wl = build_workload(name, dev, rank, args.requests if name == args.config else None)
    cu_q = None
    q_lat_s, q_pe_s = wl.q_lat, wl.q_pe  # the step's query rows
    if varlen:
        # per-request verify lengths U{1..4}: request b's queries are the first
        # q_len_b of its four query rows
        qlens = verify_qlens(wl.B, rank, wl.Qt)
        pick = torch.tensor([b * wl.Qt + t for b in range(wl.B) for t in range(int(qlens[b]))], dtype=torch.int64,
                            device=dev)
        q_lat_s = wl.q_lat[pick].contiguous()
        q_pe_s = wl.q_pe[pick].contiguous()
        cu_q = torch.from_numpy(np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)).to(dev)
    # the fp8 pool is written once (the step then writes only the last token per request)
    if wl.kind == 1:
        m.mla_cache_write(wl.w_latent, wl.w_k_pe, wl.w_slots, wl.pool, wl.kind)
        last = []
        sl = wl.seq_lens.tolist()
        start = 0
        for T in sl:
            if T:
                last.append(start + T - 1)
            start += T
        idx = torch.tensor(last, device=dev, dtype=torch.int64)
        wl.w_latent, wl.w_k_pe, wl.w_slots = wl.w_latent[idx].contiguous(), wl.w_k_pe[idx].contiguous(), wl.w_slots[idx].contiguous()
        torch.cuda.synchronize()

    cache_bytes = wl.cache_bytes()
    ctx_tokens = wl.context_tokens()
    B, Qt, Hq = wl.B, wl.Qt, wl.Hq
    R = q_lat_s.shape[0]  # query tokens of the step
    D = wl.lat_dim
    lat = D != 512
    out = torch.empty((R, Hq, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((R, Hq), dtype=torch.float32, device=dev)
    wsb = m.mla_decode_latent_workspace_bytes(B, Qt, Hq, D, 0) if lat else m.mla_decode_workspace_bytes(B, Qt, Hq, 0)
    workspace = torch.empty((wsb,), dtype=torch.uint8, device=dev)
    flush = torch.empty((256 << 20,), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    # each call's status word (and the cache write's), OR-ed over the timed
    # steps outside their events (the workspace holds only the last call's)
    status_word = workspace[:4].view(torch.int32)
    status_or = torch.zeros(1, dtype=torch.int32, device=dev)
    write_status = torch.zeros(1, dtype=torch.int32, device=dev)

    def decode(q_lat, q_pe, bt, sl, cq, o, l):
        if varlen:
            m.mla_decode_varlen(q_lat, q_pe, wl.pool, wl.kind, wl.page_size, bt, sl, cq, Qt, wl.scale, o, l, workspace)
        elif lat:
            m.mla_decode_latent(q_lat, q_pe, wl.pool, D, wl.page_size, bt, sl, Qt, wl.scale, o, l, workspace)
        else:
            m.mla_decode(q_lat, q_pe, wl.pool, wl.kind, wl.page_size, bt, sl, Qt, wl.scale, o, l, workspace)

    def write(latent_rows, kpe, slots):
        if lat:
            m.mla_cache_write_latent(latent_rows, kpe, slots, wl.pool, D, status=write_status)
        else:
            m.mla_cache_write(latent_rows, kpe, slots, wl.pool, wl.kind, status=write_status)

    # clock sampling starts before the warm-up so its start-up is over before timing
    clocks = ClockSampler(torch.cuda.current_device(), clock_csv)
    clocks.start()
    clocks.wait_first()
    for _ in range(args.warmup):
        flush.fill_(1)
        write(wl.w_latent, wl.w_k_pe, wl.w_slots)
        decode(q_lat_s, q_pe_s, wl.block_table, wl.seq_lens, cu_q, out, lse)
        # the status fold runs in the warm-up too, so its first launch (and
        # module load) is not inside the timed region
        torch.bitwise_or(status_or, status_word, out=status_or)
    torch.cuda.synchronize()
    assert m.device_status(workspace) == 0, "device-side status after warm-up"

    K = args.steps
    ev = timing_events(K, stream)
    evd = timing_events(K, stream)
    if ws_ > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.mark()
    t_wall = time.perf_counter()
    for i in range(K):
        flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        write(wl.w_latent, wl.w_k_pe, wl.w_slots)
        evd[i][0].record(stream)
        decode(q_lat_s, q_pe_s, wl.block_table, wl.seq_lens, cu_q, out, lse)
        evd[i][1].record(stream)
        ev[i][1].record(stream)
        torch.bitwise_or(status_or, status_word, out=status_or)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall
    if ws_ > 1:
        dist.barrier()
    clk = clocks.stop()
    step_times = [a.elapsed_time(b) for a, b in ev]
    step_ms = sum(step_times) / K
    dec_ms = sum(a.elapsed_time(b) for a, b in evd) / K
    assert m.device_status(workspace) == 0, "device-side status after the timed steps"

    # ---- end to end through the public API with host buffers: the step's
    # inputs travel in one packed pinned buffer (one host->device copy) and the
    # outputs come back in one (one device->host copy); the device tensors
    # handed to the calls are 256-byte-aligned views of the packed buffers
    def packed(tensors):
        offs, off = {}, 0
        for k, v in tensors.items():
            off = (off + 255) // 256 * 256
            offs[k] = off
            off += v.numel() * v.element_size()
        return offs, (off + 255) // 256 * 256

    def views(buf, offs, like):
        return {k: buf[offs[k]:offs[k] + v.numel() * v.element_size()].view(v.dtype).view(v.shape)
                for k, v in like.items()}

    src = dict(q_lat=q_lat_s, q_pe=q_pe_s, w_latent=wl.w_latent, w_k_pe=wl.w_k_pe, w_slots=wl.w_slots,
               block_table=wl.block_table, seq_lens=wl.seq_lens)
    if varlen:
        src["cu_q"] = cu_q
    in_offs, in_bytes = packed(src)
    host_in_buf = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
    for k, v in views(host_in_buf, in_offs, src).items():
        v.copy_(src[k].cpu())
    dev_in_buf = torch.empty(in_bytes, dtype=torch.uint8, device=dev)
    dev_in = views(dev_in_buf, in_offs, src)
    res = dict(out=out, lse=lse)
    out_offs, out_bytes = packed(res)
    dev_out_buf = torch.empty(out_bytes, dtype=torch.uint8, device=dev)
    dev_out = views(dev_out_buf, out_offs, res)
    host_out_buf = torch.empty(out_bytes, dtype=torch.uint8).pin_memory()
    h2d, d2h = in_bytes, out_bytes
    Ke = max(3, min(K, 200))
    eve = timing_events(Ke, stream)
    for i in range(Ke + 3):
        flush.fill_(1)
        if i >= 3:
            eve[i - 3][0].record(stream)
        dev_in_buf.copy_(host_in_buf, non_blocking=True)
        write(dev_in["w_latent"], dev_in["w_k_pe"], dev_in["w_slots"])
        decode(dev_in["q_lat"], dev_in["q_pe"], dev_in["block_table"], dev_in["seq_lens"], dev_in.get("cu_q"),
               dev_out["out"], dev_out["lse"])
        host_out_buf.copy_(dev_out_buf, non_blocking=True)
        if i >= 3:
            eve[i - 3][1].record(stream)
        torch.bitwise_or(status_or, status_word, out=status_or)
    torch.cuda.synchronize()
    e2e_ms = sum(a.elapsed_time(b) for a, b in eve) / Ke
    # the end-to-end steps computed what the device-resident steps did
    assert torch.equal(dev_out["out"], out) and torch.equal(dev_out["lse"], lse), "end-to-end outputs differ"
    status_all = int(status_or.item()) | int(write_status.item())
    if status_all:
        print(f"bench: a timed call on '{name}' reported device status {status_all:#x}", file=sys.stderr)
    res = {"name": name, "wl": wl, "cache_bytes": cache_bytes, "ctx_tokens": ctx_tokens, "step_ms": step_ms,
           "dec_ms": dec_ms, "e2e_ms": e2e_ms, "h2d": h2d, "d2h": d2h, "status_all": status_all,
           "step_times": step_times, "wall": wall, "clk": clk, "K": K}
    del out, lse, workspace, flush, dev_in_buf, dev_out_buf
    return res


def line_numbers(r, ws_, peak):
    """value, roofline and e2e of one measured workload (max over ranks)."""
    tot_bytes, step_ms_max = aggregate(r["cache_bytes"], r["step_ms"])
    _, e2e_ms_max = aggregate(r["cache_bytes"], r["e2e_ms"])
    achieved = r["cache_bytes"] / (r["dec_ms"] * 1e-3) / 1e9
    return {
        "value": round(tot_bytes / (step_ms_max * 1e-3) / 1e9, 1), "ms_per_step": round(step_ms_max, 5),
        "decode_steps_per_s": round(1e3 / step_ms_max, 1),
        "ctx_tokens_per_s": round(r["ctx_tokens"] * ws_ / (step_ms_max * 1e-3), 1),
        "achieved": achieved, "frac": achieved / peak,
        "e2e": {"value": round(tot_bytes / (e2e_ms_max * 1e-3) / 1e9, 1), "unit": "GB/s",
                "ms_per_step": round(e2e_ms_max, 5), "h2d_bytes_per_step": r["h2d"],
                "d2h_bytes_per_step": r["d2h"]},
    }


def run_gpu(args):
    import torch
    import torch.distributed as dist

    ws_, rank, local = dist_env()
    if ws_ > 1:
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    torch.cuda.set_device(local)
    dev = torch.device(f"cuda:{local}")

    from mla_latent_kv_cache_gb300 import build as mbuild
    mbuild.build()

    peak, peak_kind = measured_peaks()
    side = [] if args.side == "none" else [w for w in args.side.split(",") if w and w != args.config]
    r = measure_gpu(args.config, args, dev, rank, ws_, args.clock_csv if rank == 0 else None)
    head = line_numbers(r, ws_, peak)
    cpu = cpu_baseline(args.config, r["wl"], one_thread=True) if ws_ == 1 and not args.no_cpu and rank == 0 else None
    row_bytes = r.pop("wl").row_bytes
    side_lines = {}
    for name in side:
        torch.cuda.empty_cache()
        rs = measure_gpu(name, args, dev, rank, ws_)
        n = line_numbers(rs, ws_, peak)
        entry = {"value": n["value"], "unit": "GB/s", "ms_per_step": n["ms_per_step"],
                 "decode_steps_per_s": n["decode_steps_per_s"], "ctx_tokens_per_s": n["ctx_tokens_per_s"],
                 "roofline": {"bound": "hbm", "achieved": round(n["achieved"], 1), "peak": peak,
                              "frac": round(n["frac"], 4), "traffic": traffic_for(name),
                              "algorithmic_bytes_per_launch": rs["cache_bytes"]},
                 "e2e": n["e2e"], "config": config_dict(name, rs["ctx_tokens"], rs["cache_bytes"],
                                                        rs["wl"].row_bytes, ws_),
                 "clocks": rs["clk"], "step_times": step_time_summary(rs["step_times"]),
                 "device_status_all_steps": rs["status_all"]}
        if ws_ == 1 and not args.no_cpu and rank == 0:
            entry["cpu_baseline"] = cpu_baseline(name, rs["wl"], budget_s=4.0)
        side_lines[name] = entry
        del rs, entry
    if rank != 0:
        if ws_ > 1:
            dist.destroy_process_group()
        return
    cfg = config_dict(args.config, r["ctx_tokens"], r["cache_bytes"], row_bytes, ws_)
    if args.requests is not None:
        cfg["cut_down"] = f"first {args.requests} requests only (profiling case)"
    line = {
        "metric": METRIC, "value": head["value"], "unit": "GB/s", "n_gpus": ws_, "steps": r["K"],
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if args.config != "fp8" else "e4m3+bf16",
        "data": "synthetic (seeded N(0,1) bf16 rows, shuffled block tables, NaN-filled free slots)",
        "config": cfg,
        "decode_steps_per_s": head["decode_steps_per_s"],
        "ctx_tokens_per_s": head["ctx_tokens_per_s"],
        "pct_of_8TBps": round(100 * head["value"] / ws_ / NOMINAL_HBM_GBS, 2),
        "pct_of_measured_hbm": round(100 * head["value"] / ws_ / peak, 2),
        "roofline": {"bound": "hbm", "achieved": round(head["achieved"], 1), "peak": peak, "unit": "GB/s",
                     "frac": round(head["frac"], 4), "traffic": traffic_for(args.config),
                     "kernel": "mla_decode call (decode kernel + split-merge kernel), CUDA events",
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs: copy, read+write)",
                     "algorithmic_bytes_per_launch": r["cache_bytes"]},
        "e2e": head["e2e"],
        "gpu_launches": 3 * r["K"],
        "clocks": r["clk"],
        "wall_s_timed_region": round(r["wall"], 3),
        "step_times": step_time_summary(r["step_times"]),
        "device_status_all_steps": r["status_all"],
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if side_lines:
        line["workloads"] = side_lines
    print(json.dumps(line), flush=True)
    if ws_ > 1:
        dist.destroy_process_group()



def _gather_inputs(dev, rank=0):
    """The fp8 workload's pool, written by the cache-write kernel, and its
    prefix sums of context lengths (the gather's cu_seq_lens)."""
    import numpy as np
    import torch
    import mla_latent_kv_cache_gb300 as m
    from mla_latent_kv_cache_gb300 import workloads as W
    wl = W.fp8(device=dev, seed=6 + 1000 * rank)
    m.mla_cache_write(wl.w_latent, wl.w_k_pe, wl.w_slots, wl.pool, wl.kind)
    sl = wl.seq_lens.cpu().numpy().astype(np.int64)
    cu = torch.from_numpy(np.concatenate([[0], np.cumsum(sl)]).astype(np.int32)).to(dev)
    return wl, cu, int(sl.sum())


def gather_cpu_sample(wl, budget_s=10.0):
    """Time the oracle's gather on whole requests (in turn) for about
    `budget_s`; returns (bytes, seconds, requests, threads)."""
    import numpy as np
    import oracle
    from mla_latent_kv_cache_gb300 import workloads as W
    sl = wl.seq_lens.cpu().numpy()
    prep, done, secs, n = {}, 0, 0.0, 0
    while secs < budget_s:
        b = n % wl.B
        if b not in prep:
            c = W.compact(wl, [b])
            prep[b] = (c["pool"], c["block_table"], np.array([0, int(sl[b])], dtype=np.int32))
        pool, bt, cu = prep[b]
        t0 = time.perf_counter()
        oracle.gather_upconvert(pool, wl.page_size, bt, cu, int(sl[b]))
        secs += time.perf_counter() - t0
        done += int(sl[b]) * GATHER_BYTES_PER_TOKEN
        n += 1
    return done, secs, n, 1  # the oracle's gather is a plain loop on one thread


def run_gather(args):
    import torch
    import torch.distributed as dist

    ws_, rank, local = dist_env()
    if ws_ > 1:
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    torch.cuda.set_device(local)
    dev = torch.device(f"cuda:{local}")
    from mla_latent_kv_cache_gb300 import build as mbuild
    mbuild.build()
    import mla_latent_kv_cache_gb300 as m

    wl, cu, rows = _gather_inputs(dev, rank)
    step_bytes = rows * GATHER_BYTES_PER_TOKEN
    dst = torch.empty((rows, 576), dtype=torch.bfloat16, device=dev)
    flush = torch.empty((256 << 20,), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step(bt=wl.block_table, c=cu, out=dst):
        m.mla_gather_upconvert(wl.pool, wl.page_size, bt, c, out)

    clocks = ClockSampler(local, args.clock_csv)
    clocks.start()
    clocks.wait_first()
    for _ in range(args.warmup):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    K = min(args.steps, 1600)  # ~0.6 ms a step: about a second
    ev = timing_events(K, stream)
    if ws_ > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.mark()
    t_wall = time.perf_counter()
    for i in range(K):
        flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall
    if ws_ > 1:
        dist.barrier()
    clk = clocks.stop()
    step_times = [a.elapsed_time(b) for a, b in ev]
    step_ms = sum(step_times) / K

    # end to end: the block table and prefix sums from pinned host memory, the
    # gathered rows back to pinned host memory, every step
    h_bt = wl.block_table.cpu().pin_memory()
    h_cu = cu.cpu().pin_memory()
    h_dst = torch.empty((rows, 576), dtype=torch.bfloat16).pin_memory()
    d_bt = torch.empty_like(wl.block_table)
    d_cu = torch.empty_like(cu)
    h2d = h_bt.numel() * 4 + h_cu.numel() * 4
    d2h = rows * 576 * 2
    Ke = 10
    eve = timing_events(Ke, stream)
    for i in range(Ke + 2):
        flush.fill_(1)
        if i >= 2:
            eve[i - 2][0].record(stream)
        d_bt.copy_(h_bt, non_blocking=True)
        d_cu.copy_(h_cu, non_blocking=True)
        step(d_bt, d_cu, dst)
        h_dst.copy_(dst, non_blocking=True)
        if i >= 2:
            eve[i - 2][1].record(stream)
    torch.cuda.synchronize()
    e2e_ms = sum(a.elapsed_time(b) for a, b in eve) / Ke
    assert torch.equal(h_dst[::4096].to(dev), dst[::4096]), "end-to-end rows differ"

    tot_bytes, step_ms_max = aggregate(step_bytes, step_ms)
    _, e2e_ms_max = aggregate(step_bytes, e2e_ms)
    if rank != 0:
        if ws_ > 1:
            dist.destroy_process_group()
        return
    peak, peak_kind = measured_peaks()
    value = tot_bytes / (step_ms_max * 1e-3) / 1e9
    achieved = step_bytes / (step_ms * 1e-3) / 1e9
    line = {
        "metric": GATHER_METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws_, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(step_ms_max, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3+fp32->bf16",
        "data": "synthetic (seeded N(0,1) bf16 sources quantised by the cache-write kernel, shuffled block tables)",
        "config": {"workload": "gather", "shape": CONFIG_TEXT["gather"], "tokens": rows,
                   "bytes_per_step": step_bytes,
                   "l2": "flushed before every step (256 MiB write, outside the timed events)",
                   "step": "mla_gather_upconvert of every context token of the pool's 64 requests",
                   "parallelism": f"replicas x{ws_} (requests are independent)"},
        "tokens_per_s": round(rows * ws_ / (step_ms_max * 1e-3), 1),
        "pct_of_measured_hbm": round(100 * value / ws_ / peak, 2),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic_for("gather"),
                     "kernel": "gather_upconvert_fp8_kernel, CUDA events",
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs: copy, read+write)",
                     "algorithmic_bytes_per_launch": step_bytes},
        "e2e": {"value": round(tot_bytes / (e2e_ms_max * 1e-3) / 1e9, 1), "unit": "GB/s",
                "ms_per_step": round(e2e_ms_max, 5), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": K,
        "clocks": clk,
        "wall_s_timed_region": round(wall, 3),
        "step_times": step_time_summary(step_times),
    }
    if ws_ == 1 and not args.no_cpu:
        b, sec, n, th = gather_cpu_sample(wl)
        line["cpu_baseline"] = {"value": round(b / sec / 1e9, 4), "unit": "GB/s", "cores": th, "kind": "oracle",
                                "sample": f"{n} whole-request gathers of the gather workload "
                                          f"({b // GATHER_BYTES_PER_TOKEN} tokens, {sec:.1f} s), C oracle, one thread"}
    print(json.dumps(line), flush=True)
    if ws_ > 1:
        dist.destroy_process_group()


def run_gather_reference(args):
    """The oracle's gather as the reference arm (rank 0 only): each step whole
    requests of the gather workload, about a minute in total."""
    ws_, rank, _ = dist_env()
    if rank != 0:
        return
    import torch
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    if dev == "cuda":
        from mla_latent_kv_cache_gb300 import build as mbuild
        mbuild.build()
        wl, _, _ = _gather_inputs(dev)
    else:
        raise SystemExit("the gather workload's pool is written by the GPU cache-write kernel")
    per_step = max(0.05, 60.0 / (args.steps + args.warmup))
    tb, ts, tn = 0, 0.0, 0
    for i in range(args.warmup + args.steps):
        b, sec, n, th = gather_cpu_sample(wl, budget_s=per_step)
        if i >= args.warmup:
            tb, ts, tn = tb + b, ts + sec, tn + n
    v = tb / ts / 1e9
    print(json.dumps({
        "impl": "reference", "metric": GATHER_METRIC, "value": round(v, 4), "unit": "GB/s", "n_gpus": ws_,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * ts / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3+fp32->bf16",
        "data": "synthetic", "config": {"workload": "gather", "shape": CONFIG_TEXT["gather"]},
        "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": th, "kind": "oracle",
                         "sample": f"each step: whole requests of the gather workload for {per_step:.2f} s "
                                   f"({tn} requests over the timed steps)"},
        "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ------------------------------------------------------------ CPU oracle leg

def _oracle_prepare(wl, b):
    """Host copy of request b (its pages only, renumbered) with the step's
    new rows written by the oracle's own cache write."""
    import oracle
    from mla_latent_kv_cache_gb300 import workloads as W
    c = W.compact(wl, [b])
    pool = c["pool"].copy()
    if wl.lat_dim == 512:
        oracle.cache_write(c["w_latent"], c["w_k_pe"], c["w_slots"], pool, wl.kind)
    return c, pool


def _oracle_run(wl, prep, cap=None, qt=None):
    """Time the oracle's decode of a prepared request (its first `cap`
    tokens when given; a verify step of `qt` tokens, its first qt query rows,
    when given); returns (bytes, seconds)."""
    import numpy as np
    import oracle
    c, pool = prep
    sl = c["seq_lens"].copy()
    if cap is not None:
        sl[0] = min(int(sl[0]), int(cap))
    qt = wl.Qt if qt is None else int(qt)
    t0 = time.perf_counter()
    if wl.lat_dim != 512:
        # other latent widths: the pool as it stands (a timing sample only)
        oracle.decode_latent(c["q_lat"][:qt], c["q_pe"][:qt], pool.view(np.uint16), wl.lat_dim, 64, wl.page_size,
                             c["block_table"], sl, 1, qt, wl.Hq, wl.scale)
    else:
        oracle.decode(c["q_lat"][:qt], c["q_pe"][:qt], pool, wl.kind, wl.page_size, c["block_table"], sl, 1, qt,
                      wl.Hq, wl.scale)
    return int(sl[0]) * wl.row_bytes, time.perf_counter() - t0


def _qt_for(config, wl):
    """Per-request verify lengths of the workload (None: wl.Qt for all)."""
    return verify_qlens(wl.B, 0, wl.Qt) if config.startswith("verify") else None


def oracle_sample(config, wl, budget_s=15.0):
    """Time the oracle on whole requests of the workload (middle lengths
    first, then around again) until about `budget_s` of CPU work; returns
    (bytes, seconds, requests decoded, passes over the workload, threads)."""
    import oracle
    sl = wl.seq_lens.cpu().numpy()
    order = [int(b) for b in sorted(range(wl.B), key=lambda b: sl[b]) if sl[b] > 0]
    order = order[len(order) // 2:] + order[:len(order) // 2]
    prep = {}
    qts = _qt_for(config, wl)
    done_bytes, secs, n = 0, 0.0, 0
    while secs < budget_s:
        b = order[n % len(order)]
        if b not in prep:
            prep[b] = _oracle_prepare(wl, b)
        nb, dt = _oracle_run(wl, prep[b], qt=None if qts is None else qts[b])
        done_bytes += nb
        secs += dt
        n += 1
    return done_bytes, secs, n, n / len(order), oracle.num_threads()


def cpu_baseline(config, wl, budget_s=15.0, one_thread=False):
    """The oracle, as it stands, on whole requests of the workload for about
    `budget_s` on all host cores; with `one_thread`, also a shorter run on
    one thread (value_1_thread)."""
    import oracle
    b, s, n, passes, th = oracle_sample(config, wl, budget_s)
    d = {"value": round(b / s / 1e9, 4), "unit": "GB/s", "cores": th, "kind": "oracle",
         "sample": f"{n} whole-request decodes of the '{config}' workload ({passes:.2f} passes over its "
                   f"{int((wl.seq_lens > 0).sum())} non-empty requests, {b // wl.row_bytes} context tokens, "
                   f"{s:.1f} s), fp64 C oracle with OpenMP over (query, head)"}
    if one_thread:
        oracle.set_num_threads(1)
        try:
            b1, s1, n1, _, _ = oracle_sample(config, wl, budget_s / 5)
        finally:
            oracle.set_num_threads(th)
        d["value_1_thread"] = round(b1 / s1 / 1e9, 4)
        d["sample_1_thread"] = f"{n1} whole-request decodes, {b1 // wl.row_bytes} context tokens, {s1:.1f} s"
    return d


def run_reference(args):
    """The oracle as the reference arm: each step decodes about the same
    number of context tokens, whole requests of the workload taken in turn
    (the last one cut to the budget), so the whole run takes about a minute
    of CPU time on the host cores; rank 0 only."""
    ws_, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    import torch
    from mla_latent_kv_cache_gb300 import workloads as W
    wl = build_workload(args.config, "cuda" if torch.cuda.is_available() else "cpu")
    sl = wl.seq_lens.cpu().numpy()
    live = [int(b) for b in range(wl.B) if sl[b] > 0]
    prep = {}
    qts = _qt_for(args.config, wl)

    def run_req(b, cap=None):
        if b not in prep:
            prep[b] = _oracle_prepare(wl, b)
        return _oracle_run(wl, prep[b], cap, None if qts is None else qts[b])

    # calibrate context tokens per second on one whole request
    nb, dt = run_req(live[0])
    rate = (nb / wl.row_bytes) / max(dt, 1e-6)
    per_step = max(0.02, 60.0 / (args.steps + args.warmup))
    budget = max(16, int(rate * per_step))
    cursor = 0
    tb, ts = 0, 0.0
    for i in range(args.warmup + args.steps):
        left, sb, st = budget, 0, 0.0
        while left > 0:
            b = live[cursor % len(live)]
            cursor += 1
            take = min(int(sl[b]), left)
            nb, dt = run_req(b, take)
            left -= take
            sb += nb
            st += dt
        if i >= args.warmup:
            tb += sb
            ts += st
    v = tb / ts / 1e9
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s", "n_gpus": ws_,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * ts / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) bf16 rows, shuffled block tables, NaN-filled free slots)",
        "config": config_dict(args.config, wl.context_tokens(), wl.cache_bytes(), wl.row_bytes, ws_),
        "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": f"each step: {budget} context tokens of the '{args.config}' workload, whole "
                                   f"requests taken in turn (the last cut to the budget), all "
                                   f"{wl.Hq * wl.Qt} query rows"},
        "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=6000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default="mtp", choices=sorted(CONFIG_TEXT),
                    help="the headline workload (default: mtp, the largest one-GPU configuration)")
    ap.add_argument("--side", default=",".join(SIDE_WORKLOADS),
                    help="comma-separated workloads measured after the headline one and reported under "
                         "'workloads' in its line ('none' to skip)")
    ap.add_argument("--clock-csv", default=None, help="write the headline run's nvidia-smi clock samples here")
    ap.add_argument("--requests", type=int, default=None,
                    help="long / fp8 / mtp headline only: keep this many requests (a cut-down case for profiling; "
                         "the line then describes that case, not the named workload)")
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.config == "gather":
        run_gather_reference(args) if args.impl == "reference" else run_gather(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
