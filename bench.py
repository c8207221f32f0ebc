"""Benchmark of the quantized paged KV cache hot path.

One step = one decode layer per cache format of the Llama-3-8B-shaped
workload (32 sequences x 4096 context, 32 query / 8 KV heads, head_dim 128,
block_size 16; formats bf16, fp8 with a per-tensor scale, turbo4): for each
format, the cache write of that step's 32 new tokens (one per sequence, at
position 4095) followed by the paged decode over all 4096 positions.
The caches (956 MB in total, far above the 129 MB L2) are filled before the
timed region with the same write kernel.

value  = algorithmic bytes of the step / step time, in GB/s.  Algorithmic
         bytes = cache bytes the decode must read (every attended K/V row of
         every KV head, data + scales) + the write's input rows read and
         cache rows written.
e2e    = the same bytes / step time measured through the public API with the
         step's inputs copied from pinned host memory and the outputs copied
         back inside the timed region.
roofline: the dominant kernel (the decode kernel of the format with the
         largest share of the step) against the measured HBM copy bandwidth.
cpu_baseline: the CPU oracle (numpy) decoding a bounded sample of the same
         workload.

``--impl reference`` times the CPU oracle alone on that workload and prints
its line (the pages ship no runnable implementation).
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged-decode HBM GB/s (cache bytes read / time), us/layer, cache-write GB/s"
WORKLOAD = "llama8b"
WORKLOAD_DESC = {
    "llama8b": "llama8b decode layer: {nseq} seqs x 4096 ctx, 32 q / 8 kv heads, head_dim 128, "
               "block_size 16; one layer per format",
    "ragged": "ragged decode layer: {nseq} seqs, lengths U[512, 16384], 32 q / 8 kv heads, "
              "head_dim 128, block_size 16",
    "longctx": "long-context decode layer: {nseq} seqs x 131072, 64 q / 8 kv heads, head_dim 128, "
               "windows 0 and 4096",
    "gemma_write": "write-heavy step: 8192-token fused-QKV write (stride 16384) + decode over "
                   "{nseq} seqs x 8192, 32 q / 16 kv heads, head_dim 256",
    "tiny": "tiny: {nseq} seqs of 37/50 tokens, 4 q / 2 kv heads, head_dim 64",
    "prefill": "chunked prefill layer: {nseq} seqs x 4096 ctx, last 512 positions the new chunk "
               "(written, then attended causally), 32 q / 8 kv heads, head_dim 128, block_size 16",
    "prefill_hd256": "chunked prefill layer: {nseq} seqs x 4096 ctx, last 512 positions the new "
                     "chunk (written, then attended causally), 32 q / 16 kv heads, head_dim 256, "
                     "block_size 16",
}
# dram__bytes_read.sum + dram__bytes_write.sum per launch of the dominant
# decode launch, from the ncu capture summarised in profiles/ (None when the
# kernel changed after the capture).
TRAFFIC = {
    ("llama8b", "bf16"): 540_853_248,
    ("llama8b", "fp8"): 269_774_848,
    ("llama8b", "turbo4"): 153_500_160,
}
# dram__bytes_read.sum + dram__bytes_write.sum per launch of the dominant
# prefill launch (the slowest format of the workload), from the 1-pass ncu
# capture summarised in profiles/ (None when the kernel changed after it).
PF_TRAFFIC = {
    ("prefill", "bf16"): 190_333_952,
    ("prefill", "fp8"): 113_056_000,
    ("prefill", "turbo4"): 78_117_120,
    ("prefill_hd256", "bf16"): 667_113_984,
    ("prefill_hd256", "turbo2"): 190_637_568,
    ("prefill_hd256", "turbo8"): 423_295_232,
}
# smsp__inst_executed.sum per launch (warp-instructions) of the same capture:
# the second roofline of the decode formats that are issue bound.  Issue
# peak = 4 warp-instructions per cycle per SM (one per sub-partition) x the
# SMs x the SM clock sampled during the timed region.
WARP_INSTR = {
    ("llama8b", "bf16"): 19_621_441,
    ("llama8b", "fp8"): 24_021_319,
    ("llama8b", "turbo4"): 47_024_420,
}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        self.index = index
        self.rows = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) == 7:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[3 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.rows)}


def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def slowest_rank(values, dev):
    """Each value maxed over the ranks of the job (the job is as slow as its
    slowest rank); unchanged on one process."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t]


def parallelism(world):
    if world == 1:
        return "one GPU"
    return (f"dp{world}: a {world}x batch, sequence i on rank i mod {world} "
            "(no collective on the data path; NCCL only for the barrier and the slowest rank's time)")


def relaunch_under_torchrun(n):
    """`--gpus N` outside torchrun: run this same command as N ranks, one per
    GPU, through torch.distributed.run on this node."""
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr=127.0.0.1", f"--master-port={port}", os.path.abspath(__file__)] + sys.argv[1:]
    return subprocess.call(cmd)


def job_rate(bytes_per_rank_step, world_size, ms_per_step):
    """Whole-job throughput in GB/s: every rank processes its own units (weak
    scaling), the step lasts as long as the slowest rank."""
    return bytes_per_rank_step * world_size / (ms_per_step * 1e-3) / 1e9


def algorithmic_decode_bytes(fmt, seq_lens, nkv, hd, bs, window=0):
    from quantized_paged_kv_reshape_gb300 import ops
    per_tok = 0
    for side in (0, 1):
        per_tok += ops.block_bytes(fmt, side, bs, nkv, hd) // bs   # bytes per token (all heads)
    lens = np.asarray(seq_lens, np.int64)
    att = np.minimum(lens, window) if window > 0 else lens
    return int(att.sum()) * per_tok


def write_bytes(fmt, ntok, nkv, hd, bs, in_bytes=2):
    from quantized_paged_kv_reshape_gb300 import ops
    out = sum(ops.block_bytes(fmt, side, bs, nkv, hd) // bs for side in (0, 1)) * ntok
    return 2 * ntok * nkv * hd * in_bytes + out + 8 * ntok


# --------------------------------------------------------------------- GPU arm

def _compare(got, ref):
    """max / mean |got - ref| and the cosine of each (sequence, head) output
    row with its reference row (rows whose reference is zero are skipped)."""
    d = (got - ref).abs()
    g2, r2 = got.reshape(-1, got.shape[-1]).double(), ref.reshape(-1, ref.shape[-1]).double()
    nr = r2.norm(dim=1)
    keep = nr > 0
    cos = (g2 * r2).sum(dim=1)[keep] / (g2.norm(dim=1)[keep] * nr[keep]).clamp_min(1e-300)
    return {"max_abs": float(d.max()), "mean_abs": float(d.mean()),
            "cos_min": round(float(cos.min()), 6) if cos.numel() else None,
            "cos_mean": round(float(cos.mean()), 6) if cos.numel() else None}


def quality_report(ops, torch, ref_pools, pools, fmts, windows, q, tables, lens, nkv, bs, nseq,
                   nq, hd, mb, k_scale, v_scale, wsp, in_dtype, dev, sparse=1e-3, reps=10,
                   sample_seqs=(), samples=None):
    """Decode output of each format against the BF16-cache decode of the same
    K/V (unquantized attention; that kernel is within 2e-3 / 2e-4 of the fp64
    oracle in the parity tests), exact and with the sparse-V skip (weights
    <= 1e-3 of the running sum dropped), and the sparse-V decode time.  The
    output rows of the sequences in `sample_seqs` go to samples[(fmt,
    window)] = (exact, sparse) for the comparison with the oracle."""
    rkp, rvp = ref_pools
    rep = {"reference": "bf16-cache decode of the same K/V"
                        + ("" if in_dtype == "bf16" else " (inputs rounded to bf16)"),
           "sparse_v_threshold": sparse}
    stream = torch.cuda.current_stream()
    for win in windows:
        rws = ops.alloc_workspace(nseq, nq, nkv, hd, bs, mb, win, "bf16", device=dev)
        ref = ops.paged_decode(q, rkp, rvp, tables, lens, "bf16", nkv, bs, sliding_window=win,
                               workspace=rws)
        for f in fmts:
            kp, vp = pools[f]

            def dec(thr, f=f, kp=kp, vp=vp, win=win):
                return ops.paged_decode(q, kp, vp, tables, lens, f, nkv, bs, k_scale=k_scale,
                                        v_scale=v_scale, sliding_window=win,
                                        sparse_v_threshold=thr, workspace=wsp[(f, win)])
            exact = dec(0.0)
            sp = dec(sparse)
            dec(sparse)
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(reps)]
            for e0, e1 in evs:
                e0.record(stream)
                dec(sparse)
                e1.record(stream)
            torch.cuda.synchronize()
            us = statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs) * 1e3
            key = f if len(windows) == 1 else f"{f}@window{win}"
            if samples is not None and sample_seqs:
                idx = torch.tensor(list(sample_seqs), device=exact.device)
                samples[(f, win)] = (exact[idx].double().cpu().numpy(),
                                     sp[idx].double().cpu().numpy())
            rep[key] = {"exact": _compare(exact, ref),
                        "sparse_v": dict(_compare(sp, ref), vs_exact=_compare(sp, exact),
                                         us_per_layer=round(us, 2))}
    return rep


def time_launches(torch, fn, reps, flush, stream):
    """Median / min / p90 of `reps` CUDA-event-timed calls of fn on `stream`,
    the L2 flushed (a read of more than it holds) before each call."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    for e0, e1 in evs:
        flush.sum()      # reads more than the L2 holds: clean lines, nothing to write back
        e0.record(stream)
        fn()
        e1.record(stream)
    torch.cuda.synchronize()
    ts = sorted(e0.elapsed_time(e1) * 1e3 for e0, e1 in evs)
    return {"median_us": statistics.median(ts), "min_us": ts[0],
            "p90_us": ts[min(len(ts) - 1, (9 * len(ts)) // 10)], "launches": reps}


def sample_sequences(lens):
    """Sequences whose outputs the oracle recomputes: the shortest and the
    longest (one of them if the batch is a single length), at most one of
    more than 32768 positions."""
    lens = np.asarray(lens)
    if lens.size == 0:
        return []
    lo, hi = int(np.argmin(lens)), int(np.argmax(lens))
    if lens[hi] > 32768 or lens[lo] == lens[hi]:
        return [hi] if lens[hi] > 32768 else sorted({0, lens.size - 1})
    return sorted({lo, hi})


def host_rows(kall, vall, lens, seqs):
    """fp32 host copies [L, nkv, hd] of the K and V rows of sequences `seqs`."""
    starts = np.concatenate([[0], np.cumsum(np.asarray(lens, np.int64))])
    return {s: (kall[int(starts[s]):int(starts[s + 1])].float().cpu().numpy(),
                vall[int(starts[s]):int(starts[s + 1])].float().cpu().numpy()) for s in seqs}


def measure_workload(args, name, dev, flush, reps, want_oracle, samples):
    """Decode layers of another workload: each format's and window's layer
    time (median of `reps` launches, L2 flushed before each), its quality
    against the BF16-cache decode of the same K/V, and (for the oracle
    comparison) the sampled sequences' inputs and outputs appended to
    `samples`."""
    import torch
    from quantized_paged_kv_reshape_gb300 import ops, workloads as W

    w = W.make(name)
    nkv, nq, hd, bs, nseq = w.num_kv_heads, w.num_q_heads, w.head_dim, w.block_size, w.num_seqs
    lens_np = np.asarray(w.seq_lens, np.int64)
    tables_np = W.block_tables(w)
    mb = tables_np.shape[1]
    tables = torch.from_numpy(tables_np).to(dev)
    lens = torch.from_numpy(w.seq_lens).to(dev)
    g = torch.Generator(device=dev)
    g.manual_seed(4711)
    ntok = int(lens_np.sum())
    slots = torch.from_numpy(W.slot_mapping_for_sequences(w, tables_np)).to(dev)
    ch_k = torch.from_numpy(W.channel_scales(w, 0)).to(dev)
    ch_v = torch.from_numpy(W.channel_scales(w, 1)).to(dev)
    kall = (torch.randn((ntok, nkv, hd), generator=g, device=dev) * ch_k).to(torch.bfloat16)
    vall = (torch.randn((ntok, nkv, hd), generator=g, device=dev) * ch_v).to(torch.bfloat16)
    k_scale = float(kall.float().abs().amax()) / 448.0
    v_scale = float(vall.float().abs().amax()) / 448.0
    q = torch.randn((nseq, nq, hd), generator=g, device=dev).to(torch.bfloat16)
    fmts, windows = list(w.formats), list(w.windows)
    pools = {}
    for f in fmts:
        kp = ops.alloc_pool(w.num_blocks, f, 0, bs, nkv, hd, device=dev)
        vp = ops.alloc_pool(w.num_blocks, f, 1, bs, nkv, hd, device=dev)
        ops.cache_write(kall.view(ntok, -1), vall.view(ntok, -1), kp, vp, slots, f, nkv, hd, bs,
                        k_scale=k_scale, v_scale=v_scale)
        pools[f] = (kp, vp)
    rkp = ops.alloc_pool(w.num_blocks, "bf16", 0, bs, nkv, hd, device=dev)
    rvp = ops.alloc_pool(w.num_blocks, "bf16", 1, bs, nkv, hd, device=dev)
    ops.cache_write(kall.view(ntok, -1), vall.view(ntok, -1), rkp, rvp, slots, "bf16", nkv, hd, bs)
    seqs = sample_sequences(lens_np) if want_oracle else []
    rows = host_rows(kall, vall, lens_np, seqs)
    del kall, vall
    wsp = {(f, win): ops.alloc_workspace(nseq, nq, nkv, hd, bs, mb, win, f, device=dev)
           for f in fmts for win in windows}
    out = torch.empty((nseq, nq, hd), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    peak, _ = peaks()
    layers = {}
    for f in fmts:
        kp, vp = pools[f]
        for win in windows:
            def dec(f=f, kp=kp, vp=vp, win=win):
                ops.paged_decode(q, kp, vp, tables, lens, f, nkv, bs, out=out, k_scale=k_scale,
                                 v_scale=v_scale, sliding_window=win, workspace=wsp[(f, win)])
            for _ in range(3):
                dec()
            m = time_launches(torch, dec, reps, flush, stream)
            nbytes = algorithmic_decode_bytes(f, w.seq_lens, nkv, hd, bs, win)
            gbs = nbytes / (m["median_us"] * 1e-6) / 1e9
            key = f if len(windows) == 1 else f"{f}@window{win}"
            layers[key] = {"us_per_layer": round(m["median_us"], 2), "decode_gbs": round(gbs, 1),
                           "frac_of_peak": round(gbs / peak, 4), "cache_bytes": nbytes,
                           "us_min": round(m["min_us"], 2), "us_p90": round(m["p90_us"], 2),
                           "timing": f"median of {reps} launches, L2 flushed before each"}
    got = {}
    quality = quality_report(ops, torch, (rkp, rvp), pools, fmts, windows, q, tables, lens, nkv,
                             bs, nseq, nq, hd, mb, k_scale, v_scale, wsp, "bf16", dev,
                             sample_seqs=seqs, samples=got)
    for (f, win), (ex, sp) in got.items():
        for i, s in enumerate(seqs):
            samples.append((name, f, win, s, q[s].double().cpu().numpy(), rows[s][0], rows[s][1],
                            ex[i], sp[i]))
    del pools, rkp, rvp, wsp
    torch.cuda.empty_cache()
    return {"config": WORKLOAD_DESC[name].format(nseq=nseq), "per_layer": layers,
            "quality": quality}


def run_gpu(args):
    import torch
    from quantized_paged_kv_reshape_gb300 import ops, workloads as W
    from quantized_paged_kv_reshape_gb300 import _abi

    ws, rank, local = dist_info()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    _abi.lib()

    w = W.rank_workload(args.workload, ws, rank)
    if args.num_seqs and args.num_seqs != w.num_seqs:
        w = W.make(args.workload, num_seqs=args.num_seqs,
                   seq_lens=np.resize(w.seq_lens, args.num_seqs).astype(np.int32))
    nkv, nq, hd, bs = w.num_kv_heads, w.num_q_heads, w.head_dim, w.block_size
    nseq = w.num_seqs
    lens_np = np.asarray(w.seq_lens, np.int64)
    tables_np = W.block_tables(w)
    mb = tables_np.shape[1]
    tables = torch.from_numpy(tables_np).to(dev)
    lens = torch.from_numpy(w.seq_lens).to(dev)
    g = torch.Generator(device=dev)
    g.manual_seed(1234 + rank)
    act = torch.bfloat16 if w.in_dtype == "bf16" else torch.float32

    # K/V of every cached position, drawn on the device with the workload's
    # distribution (per-channel scale, outlier channels).
    ch_k = torch.from_numpy(W.channel_scales(w, 0)).to(dev)
    ch_v = torch.from_numpy(W.channel_scales(w, 1)).to(dev)
    ntok = int(lens_np.sum())
    slots_all = torch.from_numpy(W.slot_mapping_for_sequences(w, tables_np)).to(dev)
    kall = (torch.randn((ntok, nkv, hd), generator=g, device=dev) * ch_k).to(act)
    vall = (torch.randn((ntok, nkv, hd), generator=g, device=dev) * ch_v).to(act)
    k_scale = float(kall.float().abs().amax()) / 448.0
    v_scale = float(vall.float().abs().amax()) / 448.0
    in_bytes = 2 if act == torch.bfloat16 else 4

    fmts = args.formats.split(",") if args.formats else list(w.formats)
    windows = list(w.windows)
    pools = {}
    write_ms = {}
    for f in fmts:
        kp = ops.alloc_pool(w.num_blocks, f, 0, bs, nkv, hd, device=dev)
        vp = ops.alloc_pool(w.num_blocks, f, 1, bs, nkv, hd, device=dev)
        pools[f] = (kp, vp)
        kf, vf = kall.view(ntok, -1), vall.view(ntok, -1)
        for rep in range(3):  # fill (the last two timed: full-cache write throughput)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            # a GPU spin ahead of the start event keeps the host's enqueue of the
            # events and the launch out of the timed interval (device time only)
            torch.cuda._sleep(1_000_000)
            e0.record()
            ops.cache_write(kf, vf, kp, vp, slots_all, f, nkv, hd, bs, k_scale=k_scale,
                            v_scale=v_scale)
            e1.record()
            torch.cuda.synchronize()
            if rep:
                write_ms.setdefault(f, []).append(e0.elapsed_time(e1))

    # Step inputs: the newest token of every sequence (its last position) and
    # its query; the write-heavy workload also writes a fused-QKV prefill
    # chunk scattered over the pool.
    last = torch.from_numpy(np.cumsum(lens_np) - 1).to(dev)
    q = torch.randn((nseq, nq, hd), generator=g, device=dev).to(act)
    knew = kall[last].contiguous()
    vnew = vall[last].contiguous()
    slots_new = slots_all[last].contiguous()
    prefill = None
    if w.write_tokens:
        fused = torch.randn((w.write_tokens, w.write_row_elems), generator=g, device=dev).to(act)
        pslots = torch.from_numpy(W.scattered_slots(w.write_tokens, w.num_blocks, bs)).to(dev)
        prefill = (fused, pslots)
    outs = {f: torch.empty((nseq, nq, hd), dtype=torch.float32, device=dev) for f in fmts}
    wsp = {(f, win): ops.alloc_workspace(nseq, nq, nkv, hd, bs, mb, win, f, device=dev)
           for f in fmts for win in windows}
    # Unquantized reference for the quality report: a BF16 cache of the same
    # K/V (the workload's inputs are bf16, so this cache holds them exactly).
    ref_pools = None
    if not args.no_quality:
        rkp = ops.alloc_pool(w.num_blocks, "bf16", 0, bs, nkv, hd, device=dev)
        rvp = ops.alloc_pool(w.num_blocks, "bf16", 1, bs, nkv, hd, device=dev)
        ops.cache_write(kall.view(ntok, -1), vall.view(ntok, -1), rkp, rvp, slots_all, "bf16",
                        nkv, hd, bs)
        ref_pools = (rkp, rvp)
    want_oracle = rank == 0 and not args.no_cpu_baseline and not args.no_quality
    sample_seqs = sample_sequences(lens_np) if want_oracle else []
    kv_samples = host_rows(kall, vall, lens_np, sample_seqs)
    del kall, vall

    stream = torch.cuda.current_stream()

    def launches(q_, k_, v_, s_, fused_=None, host_out=None):
        """The step's calls in order, as (kind, key, fn): per format its cache
        write, then its decode per window."""
        seq = []
        for f in fmts:
            kp, vp = pools[f]

            def write(f=f, kp=kp, vp=vp):
                if prefill is not None:
                    fused, pslots = prefill
                    fused = fused if fused_ is None else fused_
                    ops.cache_write(fused[:, nq * hd:], fused[:, (nq + nkv) * hd:], kp, vp, pslots,
                                    f, nkv, hd, bs, key_stride=w.write_row_elems,
                                    value_stride=w.write_row_elems, k_scale=k_scale,
                                    v_scale=v_scale)
                ops.cache_write(k_.view(nseq, -1), v_.view(nseq, -1), kp, vp, s_, f, nkv, hd, bs,
                                k_scale=k_scale, v_scale=v_scale)
            seq.append(("write", f, write))
            for win in windows:
                def decode(f=f, kp=kp, vp=vp, win=win):
                    if host_out is None:
                        ops.paged_decode(q_, kp, vp, tables, lens, f, nkv, bs, out=outs[f],
                                         k_scale=k_scale, v_scale=v_scale, sliding_window=win,
                                         workspace=wsp[(f, win)])
                        return
                    # end to end: the output goes back to the host on a copy
                    # stream, overlapping the next layers' kernels; its device
                    # buffer is reused once the previous step's copy is done
                    ob, hb = host_out[(f, win)]
                    if copied.get((f, win)) is not None:
                        stream.wait_event(copied[(f, win)])
                    ops.paged_decode(q_, kp, vp, tables, lens, f, nkv, bs, out=ob,
                                     k_scale=k_scale, v_scale=v_scale, sliding_window=win,
                                     workspace=wsp[(f, win)])
                    done = torch.cuda.Event()
                    done.record(stream)
                    copy_stream.wait_event(done)
                    with torch.cuda.stream(copy_stream):
                        hb.copy_(ob, non_blocking=True)
                    ce = torch.cuda.Event()
                    ce.record(copy_stream)
                    copied[(f, win)] = ce
                seq.append(("decode", (f, win), decode))
        return seq

    def step(calls):
        for _, _, fn in calls:
            fn()

    calls = launches(q, knew, vnew, slots_new)
    for _ in range(args.warmup):
        step(calls)
    torch.cuda.synchronize()

    # The timed loop makes the calls directly, or (--graphs) replays one CUDA
    # graph per call captured from the same C-ABI calls, as a serving step
    # would.  Measured on GB300 the two agree within 2% (direct slightly
    # ahead): the host keeps ahead of the GPU either way.
    replays, launch_mode = [fn for _, _, fn in calls], "direct calls"
    if args.graphs:
        try:
            graphs = []
            for _, _, fn in calls:
                gr = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gr):
                    fn()
                graphs.append(gr)
            torch.cuda.synchronize()
            replays, launch_mode = [gr.replay for gr in graphs], "one CUDA graph per call"
            for _ in range(args.warmup):
                for r in replays:
                    r()
            torch.cuda.synchronize()
        except RuntimeError as e:  # keep the direct calls (same kernels)
            torch.cuda.synchronize()
            launch_mode = f"direct calls (graph capture failed: {str(e).splitlines()[0][:120]})"

    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in calls] for _ in range(args.steps)]
    sampler = ClockSampler(dev.index)
    if rank == 0:
        sampler.start()
        time.sleep(0.3)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(args.steps):
        for (e0, e1), r in zip(evs[i], replays):
            e0.record(stream)
            r()
            e1.record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    ms_total = t0.elapsed_time(t1)
    if ws > 1:
        torch.distributed.barrier()
    # Per-layer figures: the median of `reps` launches of each decode layer,
    # the L2 flushed before every launch.
    flush = torch.ones(64 << 20, dtype=torch.float32, device=dev)   # 256 MB
    reps = max(50, args.steps)
    med = {key: time_launches(torch, fn, reps, flush, stream)
           for kind, key, fn in calls if kind == "decode"}
    # The other decode workloads of the same kind (one GPU only).
    per_workload, extra_samples = {}, []
    if ws == 1 and args.workload == "llama8b" and not args.no_extra and not args.num_seqs:
        for name in ("ragged", "longctx"):
            per_workload[name] = measure_workload(args, name, dev, flush, reps, want_oracle,
                                                  extra_samples)
    clocks = sampler.stop() if rank == 0 else None
    ev = {key: [] for kind, key, _ in calls if kind == "decode"}
    evw = {key: [] for kind, key, _ in calls if kind == "write"}
    for i in range(args.steps):
        for (kind, key, _), pair in zip(calls, evs[i]):
            (ev if kind == "decode" else evw)[key].append(pair)

    # e2e through the public API: pinned host inputs -> device, outputs -> host.
    h_in = [t.cpu().pin_memory() for t in (q, knew, vnew, slots_new, tables, lens)]
    d_in = [torch.empty_like(t) for t in (q, knew, vnew, slots_new, tables, lens)]
    h_out = {(f, win): torch.empty((nseq, nq, hd), dtype=torch.float32).pin_memory()
             for f in fmts for win in windows}
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    if prefill is not None:
        h_fused = prefill[0].cpu().pin_memory()
        d_fused = torch.empty_like(prefill[0])
        h2d += h_fused.numel() * h_fused.element_size()
    d2h = sum(t.numel() * t.element_size() for t in h_out.values())

    copy_stream = torch.cuda.Stream(device=dev)
    copied = {}
    e2e_out = {key: (torch.empty_like(outs[key[0]]), h_out[key]) for key in h_out}
    e2e_calls = launches(d_in[0], d_in[1], d_in[2], d_in[3],
                         fused_=d_fused if prefill is not None else None, host_out=e2e_out)

    def e2e_step():
        for src, dst in zip(h_in, d_in):
            dst.copy_(src, non_blocking=True)
        if prefill is not None:
            d_fused.copy_(h_fused, non_blocking=True)
        step(e2e_calls)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e_steps = max(10, args.steps // 4)
    s0 = torch.cuda.Event(enable_timing=True)
    s1 = torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    for _ in range(e_steps):
        e2e_step()
    stream.wait_stream(copy_stream)   # every output is on the host
    s1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = s0.elapsed_time(s1) / e_steps

    ms_step, e2e_ms = slowest_rank([ms_total / args.steps, e2e_ms], dev)
    main_samples = {}
    quality = quality_report(ops, torch, ref_pools, pools, fmts, windows, q, tables, lens, nkv,
                             bs, nseq, nq, hd, mb, k_scale, v_scale, wsp, w.in_dtype, dev,
                             sample_seqs=sample_seqs, samples=main_samples) \
        if ref_pools is not None else None
    oracle_samples = [(args.workload, f, win, s, q[s].double().cpu().numpy(), kv_samples[s][0],
                       kv_samples[s][1], main_samples[(f, win)][0][i], main_samples[(f, win)][1][i])
                      for (f, win) in main_samples for i, s in enumerate(sample_seqs)]
    oracle_samples += extra_samples

    dec_bytes = {(f, win): algorithmic_decode_bytes(f, w.seq_lens, nkv, hd, bs, win)
                 for f in fmts for win in windows}
    wtok = nseq + (w.write_tokens or 0)
    step_bytes = sum(dec_bytes.values()) + sum(write_bytes(f, wtok, nkv, hd, bs, in_bytes)
                                               for f in fmts)
    peak, peak_kind = peaks()
    per_layer = {}
    for (f, win), lst in ev.items():
        us_step = statistics.mean(a.elapsed_time(b) for a, b in lst) * 1e3
        m = med[(f, win)]
        us = m["median_us"]
        gbs = dec_bytes[(f, win)] / (us * 1e-6) / 1e9
        key = f if len(windows) == 1 else f"{f}@window{win}"
        per_layer[key] = {"us_per_layer": round(us, 2), "decode_gbs": round(gbs, 1),
                          "frac_of_peak": round(gbs / peak, 4), "cache_bytes": dec_bytes[(f, win)],
                          "timing": f"median of {m['launches']} launches, L2 flushed before each",
                          "us_min": round(m["min_us"], 2), "us_p90": round(m["p90_us"], 2),
                          "us_mean_in_step": round(us_step, 2)}
    full_size = not args.num_seqs or args.num_seqs == W.make(args.workload).num_seqs
    sm_hz = (clocks or {}).get("sm_mhz") or 0.0
    if full_size and sm_hz:
        nsm = torch.cuda.get_device_properties(dev).multi_processor_count
        issue_peak = 4.0 * nsm * sm_hz * 1e6
        for key, d in per_layer.items():
            n = WARP_INSTR.get((args.workload, key))
            if n:
                rate = n / (d["us_per_layer"] * 1e-6)
                d["issue"] = {"warp_instr": n, "achieved_ginst_s": round(rate / 1e9, 1),
                              "peak_ginst_s": round(issue_peak / 1e9, 1),
                              "frac": round(rate / issue_peak, 4)}
    per_write = {}
    # The step's write on its own: a CUDA graph of 20 back-to-back calls,
    # replayed, so that host launch gaps do not count (a single small write
    # bracketed by events also measures how long the GPU waited for the host
    # to enqueue it).
    write_gpu_us = {}
    for kind, key, fn in calls:
        if kind != "write":
            continue
        try:
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr):
                for _ in range(20):
                    fn()
            gr.replay()
            torch.cuda.synchronize()
            g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            g0.record(stream)
            for _ in range(5):
                gr.replay()
            g1.record(stream)
            torch.cuda.synchronize()
            write_gpu_us[key] = g0.elapsed_time(g1) * 1e3 / 100
            del gr
        except RuntimeError:
            torch.cuda.synchronize()
    for f in fmts:
        wms = statistics.mean(write_ms[f])
        us_w = statistics.mean(a.elapsed_time(b) for a, b in evw[f]) * 1e3
        per_write[f] = {"fill_gbs": round(write_bytes(f, ntok, nkv, hd, bs, in_bytes) / (wms * 1e-3) / 1e9, 1),
                        "fill_us": round(wms * 1e3, 1), "fill_tokens": ntok,
                        "fill_timing": "device time of one full-cache write (mean of 2), "
                                       "launch queued behind a GPU spin",
                        "step_write_us": round(us_w, 2), "step_write_tokens": wtok,
                        "step_write_gpu_us": round(write_gpu_us[f], 2) if f in write_gpu_us else None,
                        "step_write_gbs": round(write_bytes(f, wtok, nkv, hd, bs, in_bytes) / (us_w * 1e-6) / 1e9, 1)}
    dom = max(per_layer, key=lambda k: per_layer[k]["us_per_layer"])
    value = job_rate(step_bytes, ws, ms_step)
    e2e_value = job_rate(step_bytes, ws, e2e_ms)
    launches_per_step = len(fmts) * ((2 if prefill is not None else 1) + len(windows))
    dom_fmt = dom.split("@")[0]
    traffic = TRAFFIC.get((args.workload, dom)) if full_size else None
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC[args.workload].format(nseq=nseq),
                   "formats": fmts, "windows": windows,
                   "l2": f"inputs larger than L2 ({sum(dec_bytes.values()) / 1e6:.0f} MB of cache per step)",
                   "parallelism": parallelism(ws),
                   "launch": launch_mode},
        "per_layer": per_layer,
        "per_workload": per_workload or None,
        "cache_write": per_write,
        "roofline": {"kernel": f"{ops.decode_kernel(dom_fmt, hd, nkv, bs)} ({dom})", "bound": "hbm",
                     "achieved": per_layer[dom]["decode_gbs"], "peak": peak, "unit": "GB/s",
                     "frac": round(per_layer[dom]["decode_gbs"] / peak, 4),
                     "traffic": traffic, "peak_kind": peak_kind + " (hbm_gbs copy)",
                     "timed": "one decode launch, CUDA events on the launch stream"},
        "e2e": {"value": round(e2e_value, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4)},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    if quality is not None:
        line["quality"] = quality
    if ws > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(seconds=args.cpu_seconds)
            if oracle_samples and line.get("quality") is not None:
                line["quality"]["vs_oracle_fp64"] = oracle_quality(oracle_samples)
        print(json.dumps(line))


# --------------------------------------------------------------------- CPU oracle

class OracleSample:
    """One sequence of the workload (``ntok`` positions x 8 kv / 32 q heads,
    turbo4) written and decoded by the CPU oracle."""

    def __init__(self, ntok=4096, fmt="turbo4"):
        import oracle
        from quantized_paged_kv_reshape_gb300 import workloads as W
        self.oracle, self.fmt = oracle, fmt
        w = W.make(WORKLOAD, num_seqs=1, seq_lens=np.array([ntok], np.int32))
        self.w = w
        nkv, hd, bs = w.num_kv_heads, w.head_dim, w.block_size
        self.tables = W.block_tables(w)
        slots = W.slot_mapping_for_sequences(w, self.tables)
        kside, vside = oracle.kv_pair(fmt)
        self.kst = oracle.block_bytes(kside, bs, nkv, hd)
        self.vst = oracle.block_bytes(vside, bs, nkv, hd)
        self.kc = np.zeros(w.num_blocks * self.kst, np.uint8)
        self.vc = np.zeros(w.num_blocks * self.vst, np.uint8)
        oracle.cache_write(kside, W.kv_rows(w, 0, ntok), self.kc, slots, nkv, hd, bs, self.kst)
        oracle.cache_write(vside, W.kv_rows(w, 1, ntok), self.vc, slots, nkv, hd, bs, self.vst)
        self.q = W.q_rows(w)
        self.nbytes = ntok * (self.kst + self.vst) // bs
        self.desc = (f"one {fmt} sequence of the workload ({ntok} tokens, 8 kv / 32 q heads, "
                     f"{self.nbytes} cache bytes)")

    def run(self):
        w = self.w
        self.oracle.paged_decode(self.q, self.kc, self.vc, self.tables, w.seq_lens,
                                 w.num_kv_heads, w.head_dim, w.block_size, self.kst, self.vst,
                                 self.fmt)


def _oracle_job(job):
    """One host process: decode its own sample sequence with the oracle after
    `warmup` untimed runs, for `reps` runs (or, if reps is 0, for `seconds`);
    returns (bytes, seconds, description)."""
    ntok, warmup, reps, seconds = job
    s = OracleSample(ntok)
    for _ in range(warmup):
        s.run()
    done, t0 = 0, time.perf_counter()
    while True:
        s.run()
        done += 1
        el = time.perf_counter() - t0
        if (reps and done >= reps) or (not reps and el >= seconds):
            break
    return done * s.nbytes, el, s.desc


def oracle_on_host_cores(ntok, warmup, reps, seconds):
    """The oracle as it stands, one single-threaded process per host core
    (a spawn pool: safe after CUDA was initialised in this process).  Returns
    (aggregate GB/s, per-process GB/s, processes, wall seconds, description)."""
    import multiprocessing as mpr
    procs = os.cpu_count() or 1
    keys = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
    saved = {k: os.environ.get(k) for k in keys}
    for k in keys:
        os.environ[k] = "1"   # inherited by the spawned processes
    try:
        with mpr.get_context("spawn").Pool(procs) as pool:
            res = pool.map(_oracle_job, [(ntok, warmup, reps, seconds)] * procs)
    except OSError:   # no processes to be had: this process alone
        procs = 1
        res = [_oracle_job((ntok, warmup, reps, seconds))]
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    wall = max(r[1] for r in res)
    total = sum(r[0] for r in res)
    per = sum(r[0] / r[1] for r in res) / procs
    return total / wall / 1e9, per / 1e9, procs, wall, res[0][2]


def oracle_quality(samples, sparse=1e-3):
    """Each format's GPU output rows of sampled sequences against the
    oracle's fp64 attention over the original (bf16) K/V of those
    sequences: max / mean |difference| and the cosine of each output row, for
    the exact decode and for the one with the sparse-V skip."""
    import oracle
    acc = {}
    for wname, fmt, win, s, q, k, v, ex, sp in samples:
        lo = max(0, k.shape[0] - win) if win > 0 else 0
        ref = oracle.attend(q, k[lo:], v[lo:])
        key = f"{wname}:{fmt}" + (f"@window{win}" if wname == "longctx" else "")
        a = acc.setdefault(key, {"exact": [], "sparse_v": [], "seqs": []})
        a["seqs"].append(int(s))
        for part, got in (("exact", ex), ("sparse_v", sp)):
            d = np.abs(got - ref)
            nr = np.linalg.norm(ref, axis=1)
            cos = (got * ref).sum(axis=1) / np.maximum(np.linalg.norm(got, axis=1) * nr, 1e-300)
            a[part].append((d.max(), d.sum(), d.size, cos[nr > 0]))
    out = {"reference": "oracle fp64 attention on the original bf16 K/V of the sampled sequences",
           "sparse_v_threshold": sparse}
    for key, a in acc.items():
        r = {"seqs": a["seqs"]}
        for part in ("exact", "sparse_v"):
            lst = a[part]
            cos = np.concatenate([x[3] for x in lst]) if lst else np.zeros(0)
            r[part] = {"max_abs": float(max(x[0] for x in lst)),
                       "mean_abs": float(sum(x[1] for x in lst) / sum(x[2] for x in lst)),
                       "cos_min": round(float(cos.min()), 6) if cos.size else None,
                       "cos_mean": round(float(cos.mean()), 6) if cos.size else None}
        out[key] = r
    return out


def cpu_baseline(seconds=15.0):
    agg, per, procs, wall, desc = oracle_on_host_cores(4096, 1, 0, seconds)
    return {"value": round(agg, 4), "unit": "GB/s", "cores": procs, "kind": "oracle",
            "per_core": round(per, 4),
            "sample": f"{procs} processes (one numpy thread each), each decoding {desc} with "
                      f"the numpy oracle repeatedly for ~{seconds:.0f} s ({wall:.1f} s wall)"}


def prefill_flops(seq_lens, chunk, nq, hd):
    """Algorithmic FLOPs of one chunked-prefill layer: query i of a chunk of C
    over L positions attends p + 1 = L - C + i + 1 keys; per key and query
    head 2*hd for q.k and 2*hd for p.v."""
    keys = sum(chunk * (int(L) - chunk) + chunk * (chunk + 1) // 2 for L in seq_lens)
    return 4 * hd * nq * keys


def run_prefill(args):
    """Chunked-prefill leg: per format, the write of every sequence's last
    `chunk` positions, then their causal attention over the paged cache."""
    import torch
    from quantized_paged_kv_reshape_gb300 import ops, workloads as W
    from quantized_paged_kv_reshape_gb300 import _abi

    ws, rank, local = dist_info()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    _abi.lib()
    w = W.rank_workload(args.workload, ws, rank)
    nkv, nq, hd, bs, C = w.num_kv_heads, w.num_q_heads, w.head_dim, w.block_size, w.chunk
    nseq = w.num_seqs
    lens_np = np.asarray(w.seq_lens, np.int64)
    tables_np = W.block_tables(w)
    tables = torch.from_numpy(tables_np).to(dev)
    lens = torch.from_numpy(w.seq_lens).to(dev)
    g = torch.Generator(device=dev)
    g.manual_seed(4321 + rank)
    ntok = int(lens_np.sum())
    slots_all = torch.from_numpy(W.slot_mapping_for_sequences(w, tables_np)).to(dev)
    ch_k = torch.from_numpy(W.channel_scales(w, 0)).to(dev)
    ch_v = torch.from_numpy(W.channel_scales(w, 1)).to(dev)
    kall = (torch.randn((ntok, nkv, hd), generator=g, device=dev) * ch_k).to(torch.bfloat16)
    vall = (torch.randn((ntok, nkv, hd), generator=g, device=dev) * ch_v).to(torch.bfloat16)
    k_scale = float(kall.float().abs().amax()) / 448.0
    v_scale = float(vall.float().abs().amax()) / 448.0
    starts = np.concatenate([[0], np.cumsum(lens_np)])
    chunk_idx = torch.from_numpy(np.concatenate([np.arange(starts[s + 1] - C, starts[s + 1])
                                                 for s in range(nseq)])).to(dev)
    kc, vc, sc = (kall[chunk_idx].contiguous(), vall[chunk_idx].contiguous(),
                  slots_all[chunk_idx].contiguous())
    cu = torch.from_numpy(np.arange(0, (nseq + 1) * C, C, dtype=np.int32)).to(dev)
    q = torch.randn((nseq * C, nq, hd), generator=g, device=dev).to(torch.bfloat16)
    fmts = args.formats.split(",") if args.formats else list(w.formats)
    pools, outs = {}, {}
    for f in fmts:
        kp = ops.alloc_pool(w.num_blocks, f, 0, bs, nkv, hd, device=dev)
        vp = ops.alloc_pool(w.num_blocks, f, 1, bs, nkv, hd, device=dev)
        ops.cache_write(kall.view(ntok, -1), vall.view(ntok, -1), kp, vp, slots_all, f, nkv, hd, bs,
                        k_scale=k_scale, v_scale=v_scale)
        pools[f] = (kp, vp)
        outs[f] = torch.empty((nseq * C, nq, hd), dtype=torch.bfloat16, device=dev)
    del kall, vall
    stream = torch.cuda.current_stream()
    ev = {f: [] for f in fmts}

    def step(record=False):
        for f in fmts:
            kp, vp = pools[f]
            ops.cache_write(kc.view(nseq * C, -1), vc.view(nseq * C, -1), kp, vp, sc, f, nkv, hd, bs,
                            k_scale=k_scale, v_scale=v_scale)
            if record:
                a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a0.record(stream)
            ops.paged_prefill(q, cu, C, kp, vp, tables, lens, f, nkv, bs, out=outs[f],
                              k_scale=k_scale, v_scale=v_scale)
            if record:
                a1.record(stream)
                ev[f].append((a0, a1))

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    sampler = ClockSampler(dev.index)
    if rank == 0:
        sampler.start()
        time.sleep(0.3)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        step(record=True)
    t1.record(stream)
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    clocks = sampler.stop() if rank == 0 else None
    ms_step, = slowest_rank([t0.elapsed_time(t1) / args.steps], dev)
    flops = prefill_flops(lens_np, C, nq, hd)
    per_layer = {}
    for f in fmts:
        us = statistics.mean(a.elapsed_time(b) for a, b in ev[f]) * 1e3
        cache_b = algorithmic_decode_bytes(f, lens_np, nkv, hd, bs)
        per_layer[f] = {"us_per_layer": round(us, 2), "tflops": round(flops / (us * 1e-6) / 1e12, 2),
                        "cache_bytes": cache_b}
    dom = max(per_layer, key=lambda k: per_layer[k]["us_per_layer"])
    pk = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    peak = pk.get("bf16_tflops") or 1900.0
    tf_step = job_rate(flops * len(fmts), ws, ms_step) / 1e3
    if rank == 0:
        print(json.dumps({
            "metric": "chunked-prefill attention TFLOP/s (algorithmic), us/layer", "value": round(tf_step, 2),
            "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16/bf16 hi+lo operands, f32 accumulate",
            "data": "synthetic",
            "config": {"workload": WORKLOAD_DESC[args.workload].format(nseq=nseq), "formats": fmts,
                       "l2": "caches far above L2 between steps",
                       "parallelism": parallelism(ws)},
            "per_layer": per_layer,
            "roofline": {"kernel": f"prefill_tc5_kernel ({dom})", "bound": "tensor",
                         "achieved": per_layer[dom]["tflops"], "peak": peak, "unit": "TFLOP/s",
                         "frac": round(per_layer[dom]["tflops"] / peak, 4),
                         "traffic": PF_TRAFFIC.get((args.workload, dom)),
                         "peak_kind": "measured bf16 dense, burst" if pk else "fallback",
                         "flops_per_layer": flops},
            "gpu_launches": 2 * len(fmts) * args.steps, "clocks": clocks}))


def run_reference(args):
    ws, rank, _ = dist_info()
    if rank != 0:
        return
    v, per, procs, wall, desc = oracle_on_host_cores(512, args.warmup, args.steps, 0.0)
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(wall / args.steps * 1e3, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "llama8b decode layer (turbo4 layer), each step a 512-token "
                                   "sample of one sequence per host core",
                       "parallelism": f"{procs} host processes"},
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": procs,
                             "kind": "oracle", "per_core": round(per, 4),
                             "sample": f"{args.steps} steps; per step each of {procs} processes "
                                       f"(one numpy thread each) decodes {desc} with the numpy "
                                       "oracle"},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="kvq", choices=["kvq", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-quality", action="store_true",
                    help="skip the quality report against a BF16 cache of the same K/V")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the ragged and long-context decode layers of the llama8b run")
    ap.add_argument("--graphs", action="store_true",
                    help="time per-call CUDA graph replays instead of direct calls")
    ap.add_argument("--num-seqs", type=int, default=0, help="override the number of sequences")
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(WORKLOAD_DESC))
    ap.add_argument("--formats", default="", help="comma list of catalogue formats (default: the workload's)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(relaunch_under_torchrun(args.gpus))
    if args.impl == "reference":
        run_reference(args)
    elif args.workload.startswith("prefill"):
        run_prefill(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
