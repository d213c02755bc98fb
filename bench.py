"""Benchmark of the paged decode step on GB300.

One step = the whole hot path of one decode step over one batch: copy-on-write block
copies (prefix workload), append (bf16) or quantise-append (int8, fp8) of each
sequence's new token, then paged decode attention (+ the partition merge).  The
default workload is the Llama-3-70B-shaped GQA batch (20 sequences x 8000 tokens) run
through 80 layers, each with its own K/V pools (80 x 655 MB = 52.4 GB resident in
HBM), its own queries and new tokens, back to back on one stream: a step is one decode
step of the whole 80-layer model's attention.  Other workloads run one layer
(`--config`, `--layers`).  Inputs are seeded and synthetic (workloads.py) and live in
HBM before the timed region; K/V pools of every workload but `tiny`, `prefix` and the
prefill chunks exceed the 126 MB L2, and those get an L2 flush before every timed step.

Prints ONE JSON line (rank 0).  `value` is whole-job effective bandwidth: the
algorithmic bytes of all steps on all ranks / the slowest rank's time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config gqa70b] [--layers L]
                  [--impl ours|reference]

--gpus N without a torchrun environment starts N local ranks itself (one per GPU,
independent replicas).  --impl reference times the CPU oracle (fp64 C, all host
cores) on a bounded sample of the same workload: the comparison baseline, not a
target.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "pa_decode effective KV HBM GB/s (% of GB300 peak) and decode tokens/s per layer"
UNIT = "GB/s"
DESCRIPTIONS = {
    "tiny": "tiny paged decode: 4 seqs, ctx {1,17,40,100}, 2/2 heads, head_dim 64, block 16",
    "mha13b": "Llama-2-13B-shaped MHA layer decode: 64 seqs, 40/40 heads, head_dim 128, block 16, "
              "ctx U[200,2048], 1-token append per seq",
    "gqa70b": "Llama-3-70B-shaped GQA layer decode: 20 seqs x 8000 tokens, 64/8 heads, head_dim 128, block 16",
    "prefix": "prefix-shared decode: 50 seqs sharing a 2000-token prefix + U[64,512] own tokens, "
              "32/8 heads, head_dim 128, block 16, COW copy of each seq's last block",
    "int8": "int8 KV decode: Llama-3-8B shape 32/8 heads, head_dim 128, block 32, 256 seqs, "
            "ctx log-uniform [128,32768], 1-token quantise+append per seq",
    "fp8": "fp8 (e4m3) KV decode: the int8 workload's shape with an fp8 cache and per-token scales",
    "verify70b": "draft verification, Llama-3-70B-shaped GQA: 20 seqs x 8000 tokens, 4 new tokens each "
                 "(causal among them), 64/8 heads, head_dim 128, block 16",
    "prefill8b": "chunked prefill, Llama-3-8B shape: 4 seqs x 512-token chunk on 3584 cached tokens, "
                 "32/8 heads, head_dim 128, block 16",
    "verify70b_fp8": "the draft-verification workload with an fp8 (e4m3) cache and per-token scales",
    "prefix_fp8": "the prefix-shared workload with an fp8 (e4m3) cache and per-token scales",
    "prefill8b_fp8": "the chunked-prefill workload with an fp8 (e4m3) cache and per-token scales",
}
FLUSH_L2 = {"tiny", "prefix", "prefix_fp8", "prefill8b", "prefill8b_fp8"}
L2_BYTES = 126 * 1024 * 1024

# dram__bytes_read.sum + dram__bytes_write.sum of one launch of the dominant kernel, from
# an ncu capture of the kernel source with this sha256 prefix (null once it changes).
NCU_TRAFFIC = {
    # decode: the single-buffered kernel for split bf16 / int8 contexts, the
    # double-buffered one for the rest, rows mode for narrow 8-bit chunks
    ("gqa70b", "14b3764a27efcdbc"): 655759104 + 4136704,
    ("mha13b", "14b3764a27efcdbc"): 1392701184 + 3305216,
    ("int8", "14b3764a27efcdbc"): 3144262400 + 5417984,
    ("fp8", "14b3764a27efcdbc"): 3144268800 + 5428992,
    ("verify70b_fp8", "14b3764a27efcdbc"): 339384320 + 5014272,
    # the tcgen05 kernel (P V issued by a row thread, padding row warps only keeping step);
    # prefill8b_fp8: every kernel of the call (pool offsets, dequantising pass, tcgen05
    # kernel), each captured cold
    ("prefill8b", "2dc02eb0952f1757"): 83980288 + 3249408,
    ("verify70b", "2dc02eb0952f1757"): 656806912 + 13232640,
    ("prefill8b_fp8", "2dc02eb0952f1757"): (5376 + 0) + (34649856 + 5105920) + (83948544 + 214784),
}


# the nominal HBM3e bandwidth of one GB300 (about 8 TB/s) and its dense bf16 tensor
# rate, beside the measured copy rate and cuBLAS rate
NOMINAL_HBM_GBS = 8000.0
NOMINAL_BF16_TFLOPS = 2250.0
# default number of layers per step: the 70B-shaped workload runs a whole model's 80
# layers (distinct pools); the others one layer
DEFAULT_LAYERS = {"gqa70b": 80}


def fragmentation_side_metric(case) -> dict:
    """KV capacity wasted by reserving each sequence's longest allowed context
    contiguously versus by paging (the pages' comparison: 60-80% against under 4%).  The
    reservation is the workload's longest context rounded up to a power of two."""
    longest = int(case.context_lens.max())
    reserve = 1 << max(0, (longest - 1).bit_length())
    f = workloads.fragmentation(case, reserve)
    return {"reserved_tokens_per_seq": reserve,
            "contiguous_waste": round(f["contiguous_waste"], 4),
            "paged_waste": round(f["paged_waste"], 4)}


def measured_peaks() -> dict:
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d.get("bf16_tflops", 1900.0)),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


def multi_kernel_source(case) -> str:
    """The source of the kernel a multi-token call runs (the library's own dispatch
    rule): the tcgen05 kernel for head_dim 128 and at least 16 (token, head) columns per
    kv head with a bf16 cache, 64 with an 8-bit one; else, for an 8-bit cache and at
    most 8 new tokens per sequence, the decode kernel in rows mode; else the mma.sync
    one."""
    qs = case.query_start.cpu()
    max_q = int((qs[1:] - qs[:-1]).max())
    if case.D == 128 and max_q * (case.Hq // case.Hkv) >= (16 if case.kv_dtype == "bf16" else 64):
        return "pa_multi_tc.cu"
    if case.kv_dtype != "bf16" and max_q <= 8:
        return "pa_decode.cu"
    return "pa_multi.cu"


def kernel_source_hash(name: str = "pa_decode.cu") -> str:
    """sha256[:16] of the CUDA source of the kernel a workload times."""
    src = ROOT / "paged_kv_cache_197_gb300" / "csrc" / name
    return hashlib.sha256(src.read_bytes()).hexdigest()[:16]


# ------------------------------------------------------- replicas across ranks
def replica_seed(seed: int, rank: int) -> int:
    """Each rank decodes its own batch of sequences (independent shards, weak scaling)."""
    return seed + 1000 * rank


def slowest_rank(values, device) -> list[float]:
    """Element-wise maximum over all ranks (the job is as slow as its slowest rank)."""
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    if torch.distributed.is_available() and torch.distributed.is_initialized() \
            and torch.distributed.get_world_size() > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def whole_job_gbs(bytes_per_step_per_rank: int, world: int, ms_per_step: float) -> float:
    """Bytes all ranks moved per step over the slowest rank's step time, in GB/s."""
    return bytes_per_step_per_rank * world / (ms_per_step * 1e-3) / 1e9


# ------------------------------------------------------------------ clock sampler
class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms in the background."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.rows.append((time.time(), parts))

    def stop(self, t0: float, t1: float) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = [r for ts, r in self.rows if t0 <= ts <= t1] or [r for _, r in self.rows]
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return float("nan")

        sm = [num(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(num(r[2]) for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------------- steps
class Layer:
    """One layer's device state: its K/V pools (and scales), queries, new tokens, output."""

    def __init__(self, k_cache, v_cache, k_scale, v_scale, q, new_key, new_value, out):
        self.k_cache, self.v_cache, self.k_scale, self.v_scale = k_cache, v_cache, k_scale, v_scale
        self.q, self.new_key, self.new_value, self.out = q, new_key, new_value, out


class Step:
    """The device buffers and the calls of one decode step of one workload, over
    `layers` layers that share the batch's block tables, lengths and slots (as the
    layers of one model do) but each hold their own cache, queries and new tokens."""

    def __init__(self, case: workloads.PagedCase, device, stream, shared_prefix=False, layers=1,
                 seed=0):
        import paged_kv_cache_197_gb300 as pa

        self.pa = pa
        self.case = case
        self.dev = device
        self.stream = stream
        c = case
        self.int8 = c.kv_dtype in ("int8", "fp8")  # quantised cache with per-token scales
        self.quant = pa.pa_quantize_kv_fp8 if c.kv_dtype == "fp8" else pa.pa_quantize_kv
        self.layers = []
        pool_shape = tuple(c.k_pool.shape)
        for li in range(layers):
            if li == 0:
                k_src, v_src, q, nk, nv = c.k_pool, c.v_pool, c.q, c.new_key, c.new_value
            else:  # the next layer: fresh values of the same shapes, same bookkeeping
                g = torch.Generator(device=device)
                g.manual_seed(seed * 1000 + li)
                rnd = lambda shape: torch.randn(shape, generator=g, device=device,  # noqa: E731
                                                dtype=torch.float32).to(torch.bfloat16)
                q, nk, nv = rnd(c.q.shape), rnd(c.new_key.shape), rnd(c.new_value.shape)
                k_src, v_src = rnd(pool_shape), rnd(pool_shape)
            if self.int8:
                N, Hkv, bs, D = pool_shape
                k_cache = torch.empty((N, Hkv, bs, D),
                                      dtype=torch.uint8 if c.kv_dtype == "fp8" else torch.int8,
                                      device=device)
                v_cache = torch.empty_like(k_cache)
                k_scale = torch.empty((N, Hkv, bs), dtype=torch.float32, device=device)
                v_scale = torch.empty_like(k_scale)
                slots = torch.arange(N * bs, dtype=torch.int64, device=device)
                rows = lambda p: p.permute(0, 2, 1, 3).reshape(N * bs, Hkv, D).contiguous()  # noqa: E731
                self.quant(rows(k_src), rows(v_src), k_cache, v_cache, k_scale, v_scale, slots,
                           stream=stream)
                torch.cuda.synchronize(device)
                if li == 0:
                    self.source = (c.k_pool.cpu(), c.v_pool.cpu())  # for the CPU baseline only
                    c.k_pool = c.v_pool = None  # the bf16 source is not part of the step
                del k_src, v_src
                torch.cuda.empty_cache()
            else:
                k_cache, v_cache, k_scale, v_scale = k_src, v_src, None, None
            self.layers.append(Layer(k_cache, v_cache, k_scale, v_scale, q, nk, nv,
                                     torch.empty_like(c.q)))
        self.max_ctx = int(c.context_lens.max())
        self.flag = torch.zeros(1, dtype=torch.int32, device=device)
        self.cow = c.cow_pairs.cpu()
        cow_launches = math.ceil(self.cow.shape[0] / 256) if self.cow.shape[0] else 0
        self.multi = c.query_start is not None  # several new tokens per sequence
        self.prefix = int(c.meta.get("prefix_tokens", 0)) if shared_prefix else 0
        if shared_prefix and not self.prefix:
            raise SystemExit("--shared-prefix needs a workload with a shared prefix")
        k0 = self.layers[0].k_cache
        if self.multi:
            self.max_q = max(c.meta["query_lens"])
            # sized for the tokens the batch holds (the 8-bit prefill pool)
            n = pa.pa_multi_token_workspace_size_for_tokens(c.S, c.q.shape[0], c.Hq, c.Hkv, c.D, c.bs,
                                                            pa.kv_dtype_of(k0), self.max_ctx, self.max_q,
                                                            int(c.context_lens.sum()))
            self.ws = torch.empty(n, dtype=torch.uint8, device=device) if n else None
            # append + attention (+ merge when split) + COW copies
            per_layer = 1 + 1 + (1 if self.ws is not None else 0) + cow_launches
        elif self.prefix:
            # one group: every sequence of the batch shares the prompt's blocks
            self.group_start = torch.tensor([0, c.S], dtype=torch.int32, device=device)
            self.group_prefix = torch.tensor([self.prefix], dtype=torch.int32, device=device)
            n = pa.pa_decode_shared_prefix_workspace_size(c.S, c.Hq, c.Hkv, c.D, c.bs,
                                                          pa.kv_dtype_of(k0),
                                                          self.max_ctx, c.S, self.prefix)
            self.ws = torch.empty(n, dtype=torch.uint8, device=device)
            # append + COW copies + setup, grouped prefix, own-token decode, merge
            per_layer = 1 + cow_launches + 4
        else:
            self.ws = pa.decode_workspace(c.q, k0, self.max_ctx)
            # append (or quantise-append) + decode (+ merge when split) + COW copies
            per_layer = 1 + 1 + (1 if self.ws is not None else 0) + cow_launches
        self.launches = per_layer * len(self.layers)

    def write_cache(self, L: Layer, new_key, new_value, slots):
        if self.cow.shape[0]:
            self.pa.pa_copy_blocks(L.k_cache, L.v_cache, self.cow, k_scale=L.k_scale,
                                   v_scale=L.v_scale, stream=self.stream)
        if self.int8:
            self.quant(new_key, new_value, L.k_cache, L.v_cache, L.k_scale, L.v_scale, slots,
                       err_flag=self.flag, stream=self.stream)
        else:
            self.pa.pa_reshape_and_cache(new_key, new_value, L.k_cache, L.v_cache, slots,
                                         err_flag=self.flag, stream=self.stream)

    def decode(self, L: Layer, q, tables, lens, out, query_start=None):
        if self.multi:
            self.pa.pa_multi_token_attention(
                out, q, L.k_cache, L.v_cache, tables, lens,
                self.case.query_start if query_start is None else query_start, self.case.scale,
                self.max_ctx, self.max_q, workspace=self.ws, k_scale=L.k_scale,
                v_scale=L.v_scale, err_flag=self.flag, stream=self.stream)
            return
        if self.prefix:
            self.pa.pa_decode_shared_prefix(out, q, L.k_cache, L.v_cache, tables, lens,
                                            self.case.scale, self.max_ctx, self.group_start,
                                            self.group_prefix, self.case.S, self.prefix,
                                            workspace=self.ws, k_scale=L.k_scale,
                                            v_scale=L.v_scale, err_flag=self.flag,
                                            stream=self.stream)
            return
        self.pa.pa_decode(out, q, L.k_cache, L.v_cache, tables, lens, self.case.scale,
                          self.max_ctx, workspace=self.ws, k_scale=L.k_scale,
                          v_scale=L.v_scale, err_flag=self.flag, stream=self.stream)

    def run(self, dec_events=None):
        """One step: every layer's append and decode in order.  dec_events, if given, is
        a (start, end) event pair recorded around the first layer's decode call only:
        an event between two kernels keeps the second from launching while the first
        drains (programmatic dependent launch), so the other layers run without."""
        c = self.case
        for li, L in enumerate(self.layers):
            self.write_cache(L, L.new_key, L.new_value, c.slot_mapping)
            if dec_events is not None and li == 0:
                dec_events[0].record(self.stream)
            self.decode(L, L.q, c.block_tables, c.context_lens, L.out)
            if dec_events is not None and li == 0:
                dec_events[1].record(self.stream)


def step_bytes(case) -> dict:
    dec = workloads.decode_algorithmic_bytes(case)
    app = workloads.append_algorithmic_bytes(case)
    cow = 0
    if case.cow_pairs.shape[0]:
        per_block = case.Hkv * case.bs * case.D * (1 if case.kv_dtype in ("int8", "fp8") else 2) * 2
        cow = case.cow_pairs.shape[0] * per_block * 2
    return {"decode": dec, "append": app, "cow": cow, "total": dec + app + cow,
            "decode_unique": workloads.decode_algorithmic_bytes(case, unique_blocks=True)}


# ------------------------------------------------------------------- our timing
def run_ours(args, rank, world, device) -> dict | None:
    stream = torch.cuda.Stream(device)
    maker = workloads.CONFIGS[args.config]
    with torch.cuda.stream(stream):
        case = maker(seed=replica_seed(args.seed, rank), device=device, poison=False)
        torch.cuda.synchronize(device)
        step = Step(case, device, stream, shared_prefix=args.shared_prefix, layers=args.layers,
                    seed=replica_seed(args.seed, rank))
    nbytes = step_bytes(case)
    n_layers = len(step.layers)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=device) \
        if args.config in FLUSH_L2 and not args.hot else None

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(device)

    sampler = ClockSampler(device.index if device.index is not None else 0)
    sampler.start()
    time.sleep(0.3)
    # warm-up: at least W steps and (unless --quick) at least half a second, so the
    # clocks settle
    t_w = time.time()
    n = 0
    settle = 0.0 if args.quick else 0.5
    while n < args.warmup or time.time() - t_w < settle:
        with torch.cuda.stream(stream):
            step.run()
        n += 1
        if n % 50 == 0:
            torch.cuda.synchronize(device)
    barrier()
    t0 = time.time()
    dec_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
    if flush is None:
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for i in range(args.steps):
            step.run(dec_ev[i])
        end.record(stream)
        barrier()
        total_ms = start.elapsed_time(end)
    else:  # flush L2 before each step, outside the timed spans
        spans = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(args.steps)]
        for i in range(args.steps):
            with torch.cuda.stream(stream):
                flush.fill_(float(i))
            spans[i][0].record(stream)
            step.run(dec_ev[i])
            spans[i][1].record(stream)
        barrier()
        total_ms = sum(a.elapsed_time(b) for a, b in spans)
    t1 = time.time()
    clocks = sampler.stop(t_w, t1)
    dec_ms = [a.elapsed_time(b) for a, b in dec_ev]
    assert int(step.flag.item()) == 0, f"kernel error flag {int(step.flag.item())}"

    # slowest rank sets the job time
    total_ms, dec_mean_ms = slowest_rank([total_ms, statistics.mean(dec_ms)], device)
    ms_per_step = total_ms / args.steps

    e2e = None if args.quick else run_e2e(args, step, case, device, stream, world)
    if rank != 0:
        return None

    peaks = measured_peaks()
    flops = workloads.multi_token_flops(case) if step.multi else 0
    if step.multi:
        kernel_name = ("pa_multi_token_attention call (attention + partition merge), kernel in "
                       + multi_kernel_source(case))
        achieved = nbytes["decode"] / (dec_mean_ms * 1e-3) / 1e9
    elif step.prefix:
        # the grouped path must move each shared block once: the unique bytes are its
        # algorithmic bytes (the per-sequence count stays in bytes_per_step)
        achieved = nbytes["decode_unique"] / (dec_mean_ms * 1e-3) / 1e9
        kernel_name = ("pa_decode_shared_prefix call (setup, grouped prefix, own-token "
                       "decode, merge); algorithmic bytes count each shared block once")
    else:
        achieved = nbytes["decode"] / (dec_mean_ms * 1e-3) / 1e9
        kernel_name = "pa_decode call (decode + partition merge)"
    src_hash = kernel_source_hash(multi_kernel_source(case) if step.multi else
                                  "pa_prefix.cu" if step.prefix else "pa_decode.cu")
    traffic = NCU_TRAFFIC.get((args.config, src_hash))
    value = whole_job_gbs(nbytes["total"] * n_layers, world, ms_per_step)
    res = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": case.kv_dtype, "data": "synthetic (seeded N(0,1))",
        "config": {"workload": DESCRIPTIONS[args.config], "name": args.config, "S": case.S,
                   "Hq": case.Hq, "Hkv": case.Hkv, "head_dim": case.D, "block_size": case.bs,
                   "pool_blocks": case.N, "total_context_tokens": int(case.context_lens.sum()),
                   "parallelism": f"replicas x{world} (independent sequence shards)",
                   "l2": "flushed before each step" if flush is not None else
                         "hot: not flushed (--hot)" if args.hot and args.config in FLUSH_L2 else
                         "K/V pools far larger than L2 (no flush needed)",
                   "layers": n_layers,
                   "bytes_per_layer": nbytes},
        # tokens attended per second and layer: one per sequence in decode, every new
        # token in a multi-token step (a step covers n_layers layers)
        "tokens_per_s_per_layer": round(case.q.shape[0] * n_layers * world / (ms_per_step * 1e-3), 1),
        "pct_of_peak": round(100 * value / world / peaks["hbm_gbs"], 2),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "traffic": traffic, "kernel": kernel_name,
                     "peak_source": peaks["source"], "mean_decode_us": round(dec_mean_ms * 1e3, 2),
                     "nominal_peak": NOMINAL_HBM_GBS,
                     "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                     "decode_calls_timed": len(dec_ms),
                     "timed_calls": "the first layer's decode call of every timed step"
                                    if n_layers > 1 else "every timed step's decode call"},
        "fragmentation": fragmentation_side_metric(case),
        "e2e": e2e,
        "gpu_launches": step.launches * args.steps,
        "clocks": clocks,
        "kernel_source": src_hash,
    }
    if n_layers > 1:
        # the whole model's attention for one decode step, measured: every layer's append
        # and decode back to back on one stream, each layer on its own pools
        res["model_step"] = {"layers": n_layers, "ms": round(ms_per_step, 4),
                             "attention_ms_estimate": round(n_layers * dec_mean_ms, 4),
                             "tokens_per_s": round(case.q.shape[0] * world / (ms_per_step * 1e-3), 1),
                             "resident_kv_gb": round(n_layers * nbytes["decode"] / 1e9, 2)}
    if step.multi:
        tflops = flops / (dec_mean_ms * 1e-3) / 1e12
        res["config"]["new_tokens_per_seq"] = step.max_q
        res["config"]["query_rows"] = int(case.q.shape[0])
        res["flops_per_step"] = flops
        res["tflops"] = round(tflops, 1)
        # bound: whichever of the two rooflines the step is closer to
        tpeak = peaks["bf16_tflops"]
        if tflops / tpeak > achieved / peaks["hbm_gbs"]:
            res["roofline"].update({"bound": "tensor", "achieved": round(tflops, 1), "peak": tpeak,
                                    "unit": "TFLOP/s", "frac": round(tflops / tpeak, 4),
                                    "peak_source": peaks["source"] + " (cuBLAS bf16 burst)",
                                    "nominal_peak": NOMINAL_BF16_TFLOPS,
                                    "frac_of_nominal": round(tflops / NOMINAL_BF16_TFLOPS, 4),
                                    "hbm_gbs": round(achieved, 1)})
        else:
            res["roofline"]["tflops"] = round(tflops, 1)
    if step.prefix:
        res["config"]["decode_path"] = "shared-prefix (one group of all sequences)"
        res["roofline"]["achieved_per_sequence_bytes"] = round(
            nbytes["decode"] / (dec_mean_ms * 1e-3) / 1e9, 1)
    elif case.shared_prefix_blocks:
        res["roofline"]["achieved_unique_bytes"] = round(
            nbytes["decode_unique"] / (dec_mean_ms * 1e-3) / 1e9, 1)
    if not args.no_cpu_baseline and not args.quick and world == 1:
        res["cpu_baseline"] = cpu_baseline(args, case, step, budget_s=args.cpu_seconds)
    return res


def pack_inputs(tensors: dict, device) -> tuple:
    """The step's input tensors laid out back to back (16-byte aligned) in one pinned
    host buffer, and device views of the same layout in one device buffer, so that a
    step's inputs cross to the GPU in a single copy."""
    offsets, size = {}, 0
    for k, t in tensors.items():
        offsets[k] = size
        size += (t.numel() * t.element_size() + 15) // 16 * 16
    host_buf = torch.empty(size, dtype=torch.uint8).pin_memory()
    dev_buf = torch.empty(size, dtype=torch.uint8, device=device)
    dev = {}
    for k, t in tensors.items():
        n = t.numel() * t.element_size()
        host_buf[offsets[k]:offsets[k] + n].copy_(t.contiguous().view(torch.uint8).reshape(-1))
        dev[k] = dev_buf[offsets[k]:offsets[k] + n].view(t.dtype).view(t.shape)
    return host_buf, dev_buf, dev, size


def run_e2e(args, step, case, device, stream, world) -> dict:
    """Same step through the public API with the step's inputs in pinned host memory:
    each step copies every layer's queries and new K/V, and the batch's slots, tables
    and lengths, to the device (one copy of a packed buffer) and reads every layer's
    output back, all inside the timed region.  The K/V caches are resident state, like
    weights."""
    tensors = {k: getattr(case, k).cpu() for k in ("slot_mapping", "block_tables", "context_lens")}
    if step.multi:
        tensors["query_start"] = case.query_start.cpu()
    for li, L in enumerate(step.layers):
        for k in ("q", "new_key", "new_value"):
            tensors[f"{k}{li}"] = getattr(L, k).cpu()
    host_buf, dev_buf, dev, h2d = pack_inputs(tensors, device)
    outs = torch.empty((len(step.layers),) + tuple(case.q.shape), dtype=case.q.dtype, device=device)
    out_host = torch.empty(outs.shape, dtype=case.q.dtype).pin_memory()
    d2h = out_host.numel() * out_host.element_size()
    steps = max(3, min(args.steps, 200))

    def one():
        dev_buf.copy_(host_buf, non_blocking=True)
        for li, L in enumerate(step.layers):
            step.write_cache(L, dev[f"new_key{li}"], dev[f"new_value{li}"], dev["slot_mapping"])
            step.decode(L, dev[f"q{li}"], dev["block_tables"], dev["context_lens"], outs[li],
                        query_start=dev.get("query_start"))
        out_host.copy_(outs, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(3):
            one()
        torch.cuda.synchronize(device)
        if world > 1:
            torch.distributed.barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            one()
        b.record(stream)
        torch.cuda.synchronize(device)
    ms = slowest_rank([a.elapsed_time(b) / steps], device)[0]
    total = step_bytes(case)["total"] * len(step.layers)
    return {"value": round(whole_job_gbs(total, world, ms), 2), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 5),
            "steps": steps, "h2d_copies_per_step": 1}


# ----------------------------------------------------------------- CPU baseline
def oracle_sample_inputs(case, step=None):
    """Host copies of the caches (bf16 bits, or int8 codes and scales) for the oracle."""
    import numpy as np

    def bits(t):
        return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)

    if case.kv_dtype in ("int8", "fp8"):
        import oracle

        orc = oracle.load()
        k_src, v_src = step.source if step is not None else (case.k_pool, case.v_pool)
        kc, ks = orc.quantize_pool(bits(k_src), fp8=case.kv_dtype == "fp8")
        vc, vs = orc.quantize_pool(bits(v_src), fp8=case.kv_dtype == "fp8")
        return bits(case.q), kc, vc, ks, vs
    return bits(case.q), bits(case.k_pool), bits(case.v_pool), None, None


def first_sequences(case, n):
    """The case cut to its first n sequences (for byte accounting of a sample)."""
    sub = workloads.PagedCase(**{**case.__dict__})
    sub.S = n
    sub.context_lens = case.context_lens[:n].cpu()
    sub.block_tables = case.block_tables[:n].cpu()
    if case.query_start is not None:
        qs = case.query_start.cpu()
        sub.query_start = qs[: n + 1]
        sub.q = case.q[: int(qs[n])]
    else:
        sub.q = case.q[:n]
    return sub


def oracle_runner(orc, case, inputs):
    """A call of the oracle over the first n sequences of the case."""
    import numpy as np

    q, kc, vc, ks, vs = inputs
    tables = case.block_tables.cpu().numpy()
    lens = case.context_lens.cpu().numpy()
    if case.query_start is None:
        return lambda n: orc.paged_attention(
            np.ascontiguousarray(q[:n]), kc, vc, np.ascontiguousarray(tables[:n]),
            np.ascontiguousarray(lens[:n]), case.scale, k_scale=ks, v_scale=vs)
    qs = case.query_start.cpu().numpy()
    return lambda n: orc.paged_prefill(
        np.ascontiguousarray(q[: qs[n]]), kc, vc, np.ascontiguousarray(tables[:n]),
        np.ascontiguousarray(lens[:n]), np.ascontiguousarray(qs[: n + 1]), case.scale,
        k_scale=ks, v_scale=vs)


def time_oracle(case, inputs, budget_s: float, threads: int | None = None) -> dict:
    """Oracle decode over the first n sequences, n grown until the run takes ~budget_s
    (on `threads` host threads, default all)."""
    import oracle

    orc = oracle.load()
    all_threads = orc.num_threads
    if threads is not None:
        orc.set_num_threads(threads)
    n, elapsed = 1, 0.0
    run = oracle_runner(orc, case, inputs)
    while True:
        t0 = time.perf_counter()
        run(n)
        elapsed = time.perf_counter() - t0
        if elapsed >= budget_s / 4 or n >= case.S:
            break
        n = min(case.S, max(n + 1, int(n * min(8.0, (budget_s / 4) / max(elapsed, 1e-3)))))
    # repeat the sample until about budget_s of CPU time is spent; report the mean
    reps, total = 1, elapsed
    while total < budget_s:
        t0 = time.perf_counter()
        run(n)
        total += time.perf_counter() - t0
        reps += 1
    elapsed = total / reps
    sub = first_sequences(case, n)
    nbytes = workloads.decode_algorithmic_bytes(sub)
    what = "multi-token attention" if case.query_start is not None else "decode"
    cores = orc.num_threads
    if threads is not None:
        orc.set_num_threads(all_threads)
    return {"value": round(nbytes / elapsed / 1e9, 4), "unit": UNIT, "cores": cores,
            "kind": "oracle", "seconds": round(elapsed, 3), "repeats": reps, "sequences": n,
            "sample": f"{what} of the first {n} of {case.S} sequences "
                      f"({int(sub.context_lens.sum())} context tokens), fp64 C oracle, "
                      f"caches resident in host memory"}


def cpu_baseline(args, case, step, budget_s=20.0) -> dict:
    """The oracle on all host cores, with its single-core figure beside it."""
    inputs = oracle_sample_inputs(case, step)
    res = time_oracle(case, inputs, budget_s)
    one = time_oracle(case, inputs, budget_s / 2, threads=1)
    res["single_core"] = {"value": one["value"], "cores": one["cores"], "sample": one["sample"]}
    return res


def run_reference(args, rank, world) -> dict | None:
    """The oracle as it stands, on the host cores, over a fixed sample of the workload.

    The sample (the first n sequences) is sized once so that W + K steps take about
    two minutes in all, at most 3 s a step."""
    import oracle

    if rank != 0:
        return None
    case = workloads.CONFIGS[args.config](seed=args.seed, device="cpu", poison=False)
    inputs = oracle_sample_inputs(case)
    oracle.load().set_num_threads(os.cpu_count() or 1)  # a launcher may have set one thread
    per_step = min(3.0, 120.0 / (args.warmup + args.steps))
    info = time_oracle(case, inputs, budget_s=4 * per_step)  # calibrates n
    n = info["sequences"]
    orc = oracle.load()
    run = oracle_runner(orc, case, inputs)
    nbytes = workloads.decode_algorithmic_bytes(first_sequences(case, n))
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        run(n)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    ms_per_step = 1e3 * sum(times) / len(times)
    value = round(nbytes / (ms_per_step * 1e-3) / 1e9, 4)
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1))",
            "config": {"workload": DESCRIPTIONS[args.config], "name": args.config},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": info["cores"], "kind": "oracle",
                             "sample": info["sample"]},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def free_port() -> int:
    import socket

    with socket.socket() as sock:
        sock.bind(("127.0.0.1", 0))
        return sock.getsockname()[1]


def launch_ranks(n: int, argv: list[str]) -> int:
    """Run this script as n local ranks (torch.distributed.run, rendezvous on
    127.0.0.1) and return their exit status."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr=127.0.0.1", f"--master-port={free_port()}", str(Path(__file__).resolve()),
           *argv]
    return subprocess.run(cmd, cwd=str(ROOT)).returncode


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default="gqa70b", choices=sorted(workloads.CONFIGS))
    ap.add_argument("--layers", type=int, default=None,
                    help="layers per step, each with its own K/V pools (default: 80 for gqa70b, "
                         "1 otherwise)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=1)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--hot", action="store_true",
                    help="no L2 flush between steps for the workloads that fit in L2 (the "
                         "cached figure beside the default flushed one)")
    ap.add_argument("--shared-prefix", action="store_true",
                    help="decode through pa_decode_shared_prefix (workloads with a shared prefix)")
    ap.add_argument("--quick", action="store_true",
                    help="exactly W warm-up steps, no end-to-end or CPU legs (for profiler runs)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.layers is None:
        args.layers = DEFAULT_LAYERS.get(args.config, 1)
    if args.layers < 1:
        ap.error("--layers must be at least 1")

    if args.gpus < 1:
        ap.error("--gpus must be at least 1")
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        # one rank per GPU: start them here, as torchrun would
        sys.exit(launch_ranks(args.gpus, sys.argv[1:]))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world != args.gpus:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE is {world}: launch one rank per GPU")
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=device)
    try:
        res = run_ours(args, rank, world, device)
        if res is not None:
            print(json.dumps(res), flush=True)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
