"""Benchmark: paged decode attention KV GB/s (+ prefill TFLOP/s) on GB300.

One step = the decode hot path over one batch of the batched-decode workload
(256 sequences, context_lens uniform in [512, 4096], 16 q / 8 kv heads,
head_dim 128, block_size 256, 8192-block pool with shuffled block tables):
pkv_store_kvcache of the 256 new tokens, then pkv_decode (split-KV, merge in
the same launch). ``value`` = live K/V bytes read by the decode (each live
element once) / step time, inputs resident in HBM (2.4 GB of K/V per step,
larger than L2).

Also reported on the same line:
  roofline      decode kernel: algorithmic bytes / its CUDA-event time vs the
                measured HBM copy bandwidth (MEASURED_PEAKS.json)
  e2e           the same metric through the C ABI with host buffers: pinned
                inputs copied in, result copied out, inside the timed region
  prefill       varlen prefill (64 prompts, 100..1024 tokens, <=16384 per call)
                and prefix-cached prefill (128 seqs x 1024-token shared prefix
                + 64..512 suffix): TFLOP/s of causally live pairs, vs the
                measured bf16 dense peak; store GB/s at prefill size
  cpu_baseline  the oracle (fp64 C, OpenMP) on a bounded sample, host cores

``--impl reference`` times the oracle itself as the reference arm.
Multi-GPU: replicas only (the path has no exchange step); each rank runs the
same workload on its own GPU and value sums over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "paged decode attn KV GB/s & prefill attn TFLOPS (1xGB300, % roofline)"
UNIT = "GB/s"


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs"), d.get("bf16_tflops"), d.get("bf16_tflops_sustained"), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def _src_hash(name):
    """sha256 prefix of a kernel's source file plus the device header it includes."""
    h = hashlib.sha256()
    for part in (name, "pkv_common.cuh"):
        with open(os.path.join(ROOT, "paged_kv_cache_kvh_gb300", "csrc", part), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _traffic(kernel_file, units_now, case=None):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current source of the kernel (else None). Scaled by units processed
    when the capture used a smaller case of the same kernel; ``case`` picks a
    capture taken on one specific workload (no scaling across workloads)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel_file)
    if not e or e.get("src_sha") != _src_hash(kernel_file):
        return None
    if case is not None:
        c = e.get("cases", {}).get(case)
        return None if c is None else c["dram_bytes_per_launch"]
    return e["dram_bytes_per_launch"] * (units_now / e["units"]) if e.get("units") else e["dram_bytes_per_launch"]


def _traffic_launch(kernel_file, case):
    """Which launch of a workload a per-workload capture measured."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        c = json.load(f).get(kernel_file, {}).get("cases", {}).get(case)
    return None if c is None else c.get("launch")


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.proc = None
        self.index = index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def _make_flush(dev):
    """Two 256 MB buffers (L2 is 129 MB): one written, one read, per flush."""
    return (torch.empty(256 << 20, dtype=torch.uint8, device=dev),
            torch.ones(64 << 20, dtype=torch.float32, device=dev))


def _flush_l2(flush):
    """Write a buffer larger than L2, then read another one: L2 ends up holding
    only clean lines of the read buffer, so the next timed kernel starts cold
    and pays no write-back of the flush's dirty lines."""
    w, r = flush
    w.zero_()
    r.sum()


def _prequeue(ms):
    """Occupy the GPU for about `ms` milliseconds with a spin kernel, so the
    host can queue the launches that follow before the GPU reaches them: the
    events around each timed launch then see the kernel alone, not host-side
    launch latency (Python argument checks, tensor-map encoding) during which
    an idle GPU would wait."""
    torch.cuda._sleep(int(ms * 2.2e6))  # about 2.2e6 SM cycles per ms at the 2.07 GHz maximum clock


def _sm_count():
    return torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count


def _decode_kernel(num_seqs, max_context_len=W.MAX_MODEL_LEN):
    """The decode kernel the library launches for these sizes (its rule: whole
    256-token chunks, i.e. num_seqs * ceil(max_ctx / 256) >= 608, and at most
    512 sequences take the persistent form)."""
    whole = num_seqs * (-(-max_context_len // W.BLOCK_SIZE)) >= 608
    return "decode_persistent_kernel" if whole and num_seqs <= 512 else "decode_split_kernel"


def _prefill_kernel(num_items, max_seqlen_k):
    """The prefill kernel the library launches for a planned call (its rule:
    at least two (item, kv head) units per SM and keys <= 4096)."""
    persistent = 8 * num_items >= 2 * _sm_count() and max_seqlen_k <= 4096
    return ("prefill_persistent_kernel", "prefill_persistent.cu") if persistent else ("prefill_tc_kernel",
                                                                                       "prefill.cu")


def max_over_ranks(ms, world, device):
    """Slowest rank's time: every rank does the same work (replicas)."""
    if world <= 1:
        return float(ms)
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, world, ms_step):
    """Whole-job units per second: all ranks' units over the slowest rank's step time."""
    return world * units_per_rank / (ms_step * 1e-3)


# ---------------------------------------------------------------------------
# the decode step (ours)
# ---------------------------------------------------------------------------

def decode_case(pkv, dev, seed=2, dtype=torch.bfloat16):
    wl = W.batched_decode(seed=seed)
    gen = W.make_generator(seed, dev)
    shape = (wl.num_blocks, W.BLOCK_SIZE, W.HKV, W.HEAD_DIM)
    kc, vc = W.normal(shape, gen, dev, dtype), W.normal(shape, gen, dev, dtype)
    B = len(wl.seqs)
    qkv, q, k, v = W.fused_qkv(B, gen, dev, dtype=dtype)
    meta = pkv.metadata.prepare_decode(wl.seqs, W.BLOCK_SIZE, table_width=W.MAX_MODEL_LEN // W.BLOCK_SIZE)
    c = dict(wl=wl, kc=kc, vc=vc, qkv=qkv, q=q, k=k, v=v, meta=meta, B=B,
             slot=torch.from_numpy(meta["slot_mapping"]).to(dev),
             ctx=torch.from_numpy(meta["context_lens"]).to(dev),
             bt=torch.from_numpy(meta["block_tables"]).to(dev),
             ws=pkv.decode_workspace(B, W.MAX_MODEL_LEN, dev),
             out=torch.empty(B, W.HQ, W.HEAD_DIM, dtype=dtype, device=dev))
    ctx = meta["context_lens"].astype(np.int64)
    c["kv_bytes"] = int(ctx.sum()) * W.HKV * W.HEAD_DIM * 2 * 2
    c["decode_alg_bytes"] = (c["kv_bytes"] + B * W.HQ * W.HEAD_DIM * 2 * 2 + meta["block_tables"].nbytes
                             + B * 4)
    return c


def run_ours(args, rank, world, dev):
    import paged_kv_cache_kvh_gb300 as pkv

    c = decode_case(pkv, dev)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        pkv.pkv_store_kvcache(c["k"], c["v"], c["kc"], c["vc"], c["slot"])
        if ev is not None:
            ev[0].record(stream)
        pkv.pkv_decode(c["q"], c["kc"], c["vc"], c["bt"], c["ctx"], W.MAX_MODEL_LEN, W.SCALE, c["ws"],
                       out=c["out"])
        if ev is not None:
            ev[1].record(stream)

    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop() if sampler else None
    dec_ms = sum(a.elapsed_time(b) for a, b in evs) / args.steps
    ms_total = max_over_ranks(t0.elapsed_time(t1), world, dev)
    ms_step = ms_total / args.steps
    err = pkv.pkv_device_error()
    if err:
        raise RuntimeError(f"device error word {err:#x} after the timed region")

    # ---- e2e: host buffers through the C ABI ----
    e2e = run_e2e(pkv, c, args, dev, world)

    hbm, bf16, bf16_sus, src = _peaks()
    ach = c["decode_alg_bytes"] / (dec_ms * 1e-3) / 1e9
    roof = {"kernel": _decode_kernel(c["B"]), "bound": "hbm", "achieved": round(ach, 1), "peak": hbm,
            "unit": "GB/s", "frac": round(ach / hbm, 4), "peak_source": f"{src} (hbm copy)",
            "alg_bytes_per_launch": c["decode_alg_bytes"], "avg_launch_ms": round(dec_ms, 5),
            "traffic": _traffic("decode.cu", c["kv_bytes"])}
    res = {"metric": METRIC, "value": round(job_throughput(c["kv_bytes"], world, ms_step) / 1e9, 1), "unit": UNIT,
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
           "data": "synthetic (seeded N(0,1) bf16, shuffled block tables)",
           "config": {"workload": "batched_decode_b256_ctx512-4096: store_kvcache(256 tokens) + GQA decode",
                      "num_seqs": c["B"], "q_heads": W.HQ, "kv_heads": W.HKV, "head_dim": W.HEAD_DIM,
                      "block_size": W.BLOCK_SIZE, "num_blocks": c["wl"].num_blocks,
                      "sum_context_lens": int(c["meta"]["context_lens"].sum()),
                      "kv_bytes_per_step": c["kv_bytes"],
                      "l2": "inputs larger than L2 (2.4 GB of live K/V read per step)",
                      "parallelism": f"replicas x{world}",
                      "why_this_workload": "the metric names no workload; the value is one batched decode "
                                           "step (the listed decode-step workload), the 28-layer graph sweep "
                                           "and the prefill/store cases are reported beside it (sweep, "
                                           "prefill, store, rooflines)"},
           "roofline": roof, "e2e": e2e, "gpu_launches": 2 * args.steps, "clocks": clocks}
    rooflines = [_roof_entry(roof, "batched_decode_b256 (headline step)", "bf16")]
    if rank == 0:
        res["fused_step"] = run_fused_step(pkv, c, args)
    del c
    if rank == 0 and not args.no_prefill:
        detail = run_prefill(pkv, args, dev, bf16)
        res["prefill_detail"] = detail
        store = run_store_stream(pkv, args, dev, hbm)
        res["store"] = store
        res["prefill"] = _prefill_summary(detail, store, bf16, hbm)
        for short, name in _PREFILL_SHORT.items():
            if name in detail:
                rooflines.append(_roof_entry(detail[name]["roofline"], short, "bf16"))
        rooflines.append(_roof_entry(store["roofline"], store["roofline"]["workload"], "bf16"))
    if rank == 0:
        res["tiny_decode"] = run_tiny(pkv, args, dev)
    if rank == 0 and not args.no_sweep:
        res["sweep"] = run_sweep(pkv, args, dev, hbm)
        res["padded_graph"] = run_padded_graph(pkv, args, dev, hbm)
        sw, pg = res["sweep"], res["padded_graph"]
        rooflines.append({"kernel": _decode_kernel(512) + " (store fused)", "workload": "sweep_28l_b512 graph",
                          "dtype": "bf16", "achieved": sw["fused_store_decode"]["kv_gbs"], "peak": hbm,
                          "unit": "GB/s", "frac": sw["fused_store_decode"]["frac_of_hbm"], "traffic": None})
        rooflines.append({"kernel": _decode_kernel(256), "workload": "padded_b200_in_graph256", "dtype": "bf16",
                          "achieved": pg["live_kv_gbs"], "peak": hbm, "unit": "GB/s", "frac": pg["frac_of_hbm"],
                          "traffic": None})
    if rank == 0 and not args.no_f16:
        res["f16"] = run_f16(pkv, args, dev, hbm, bf16)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(budget_s=args.cpu_seconds)
    # last on the line, so a reader that keeps only the end of the output
    # still sees every kernel's fraction of its roofline
    res["rooflines"] = rooflines
    return res


_PREFILL_SHORT = {"prefill_varlen_64p": "varlen_prefill_64p_len100-1024",
                  "prefill_prefix_128s": "prefix_prefill_128s_prefix1024_suffix64-512",
                  "prefill_chunked_16p": "chunked_prefill_16p_len4096-12288_budget5000"}


def _roof_entry(roof, workload, dtype):
    """One flat roofline record: kernel, workload, achieved / peak, traffic."""
    return {"kernel": roof["kernel"], "workload": workload, "dtype": dtype, "achieved": roof["achieved"],
            "peak": roof["peak"], "unit": roof["unit"], "frac": roof["frac"], "traffic": roof.get("traffic")}


def _prefill_summary(detail, store, bf16_peak, hbm_peak):
    """The bf16 prefill and store figures as flat numbers (TFLOP/s of causally
    live pairs and fraction of the bf16 dense peak; store GB/s over >4 GB of
    back-to-back stores and fraction of HBM)."""
    out = {"unit": "TFLOP/s", "peak_tflops": bf16_peak}
    for short, name in (("varlen", "varlen_prefill_64p_len100-1024"),
                        ("prefix", "prefix_prefill_128s_prefix1024_suffix64-512"),
                        ("chunked", "chunked_prefill_16p_len4096-12288_budget5000")):
        if name in detail:
            out[f"{short}_tflops"] = detail[name]["tflops"]
            out[f"{short}_frac"] = detail[name]["roofline"]["frac"]
    out["store_gbs"] = store["roofline"]["achieved"]
    out["store_frac_of_hbm"] = store["roofline"]["frac"]
    out["hbm_peak_gbs"] = hbm_peak
    return out


def run_store_stream(pkv, args, dev, hbm_peak, n_calls=32, tokens=W.MAX_NUM_BATCHED_TOKENS):
    """store_kvcache at prefill size on HBM: n_calls back-to-back calls of
    `tokens` tokens each (the scheduler's per-step token cap), every call
    reading its own rows of a fused qkv buffer and writing its own shuffled
    blocks of a 2 GB pool, timed together. 4.3 GB are written per pass, so at
    most the last ~0.13 GB (one L2) can still sit in L2 when the events close;
    L2 is flushed before every pass."""
    blocks_per_call = tokens // W.BLOCK_SIZE
    nb = n_calls * blocks_per_call
    gen = W.make_generator(31, dev)
    shape = (nb, W.BLOCK_SIZE, W.HKV, W.HEAD_DIM)
    kc, vc = torch.empty(shape, dtype=torch.bfloat16, device=dev), torch.empty(shape, dtype=torch.bfloat16, device=dev)
    qkv, _, k, v = W.fused_qkv(n_calls * tokens, gen, dev)
    perm = np.random.default_rng(31).permutation(nb).reshape(n_calls, blocks_per_call)
    slots = (perm[:, :, None] * W.BLOCK_SIZE + np.arange(W.BLOCK_SIZE)[None, None, :]).reshape(n_calls, tokens)
    slot = torch.from_numpy(slots.astype(np.int32)).to(dev)
    flush = _make_flush(dev)

    def one_pass():
        for i in range(n_calls):
            pkv.pkv_store_kvcache(k[i * tokens:(i + 1) * tokens], v[i * tokens:(i + 1) * tokens], kc, vc, slot[i])

    one_pass()
    reps = max(3, min(args.steps, 10))
    evs = []
    for it in range(reps + 1):
        _prequeue(0.1 * n_calls + 1.0)
        _flush_l2(flush)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        one_pass()
        b.record()
        if it >= 1:
            evs.append((a, b))
    torch.cuda.synchronize()
    if pkv.pkv_device_error():
        raise RuntimeError("device error word set by the store stream")
    # spot check: the last call's rows landed where its slots say
    i = n_calls - 1
    got = kc.view(-1, W.HKV, W.HEAD_DIM)[slot[i, :64].long()]
    if not torch.equal(got, k[i * tokens:i * tokens + 64]):
        raise RuntimeError("store stream: rows not at their slots")
    ms = sum(x.elapsed_time(y) for x, y in evs) / len(evs)
    alg = n_calls * tokens * W.HKV * W.HEAD_DIM * 2 * 4          # read K, V + write K, V
    gbs = alg / (ms * 1e-3) / 1e9
    del kc, vc, qkv, k, v, flush
    torch.cuda.empty_cache()
    return {"workload": f"{n_calls} back-to-back store_kvcache calls x {tokens} tokens (2 GB pool)",
            "ms_per_pass": round(ms, 4), "us_per_call": round(ms * 1e3 / n_calls, 2), "passes": len(evs),
            "roofline": {"kernel": "store_kvcache_v16_kernel", "workload": f"store_{n_calls}x{tokens}tok",
                         "bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                         "frac": round(gbs / hbm_peak, 4), "alg_bytes_per_pass": alg, "traffic": None,
                         "traffic_note": "4.3 GB written per pass against a 129 MB L2: the algorithmic bytes "
                                         "reach HBM up to <= 3%"}}


def run_fused_step(pkv, c, args):
    """The headline batch's store + decode as one launch (pkv_store_decode, the
    new token's K/V written by the CTA that streams its block), device-resident
    inputs, CUDA events around `steps` back-to-back steps."""
    def step():
        pkv.pkv_store_decode(c["q"], c["k"], c["v"], c["slot"], c["kc"], c["vc"], c["bt"], c["ctx"],
                             W.MAX_MODEL_LEN, W.SCALE, c["ws"], out=c["out"])

    for _ in range(args.warmup):
        step()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record()
    for _ in range(args.steps):
        step()
    b.record()
    torch.cuda.synchronize()
    if pkv.pkv_device_error():
        raise RuntimeError("device error word set by the fused step")
    ms = a.elapsed_time(b) / args.steps
    return {"ms_per_step": round(ms, 5), "kv_gbs": round(c["kv_bytes"] / (ms * 1e-3) / 1e9, 1),
            "gpu_launches_per_step": 1, "note": "same batch and bytes as the headline step, one launch"}


def run_e2e(pkv, c, args, dev, world=1):
    """Store + decode from pinned host buffers: every step copies its inputs
    host-to-device and reads its output back. Two device input/output sets and
    separate copy streams let step k+1's copies overlap step k's kernels (the
    way a serving loop would issue them); each step still moves all its bytes.
    With several ranks the value is the whole job's, like the headline's:
    all ranks' bytes over the slowest rank's time, barriers on both sides."""
    B = c["B"]
    hq = c["q"].contiguous().cpu().pin_memory()
    hk = c["k"].contiguous().cpu().pin_memory()
    hv = c["v"].contiguous().cpu().pin_memory()
    hslot = torch.from_numpy(c["meta"]["slot_mapping"]).pin_memory()
    hctx = torch.from_numpy(c["meta"]["context_lens"]).pin_memory()
    hbt = torch.from_numpy(c["meta"]["block_tables"]).pin_memory()
    hout = [torch.empty(B, W.HQ, W.HEAD_DIM, dtype=c["out"].dtype).pin_memory() for _ in range(2)]
    sets = [dict(q=torch.empty_like(hq, device=dev), k=torch.empty_like(hk, device=dev),
                 v=torch.empty_like(hv, device=dev), slot=torch.empty_like(c["slot"]),
                 ctx=torch.empty_like(c["ctx"]), bt=torch.empty_like(c["bt"]), out=torch.empty_like(c["out"]))
            for _ in range(2)]
    comp = torch.cuda.current_stream()
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def step(k):
        i = k % 2
        S = sets[i]
        h2d.wait_event(ev_done[i])            # step k-2 no longer reads this input set
        with torch.cuda.stream(h2d):
            for name, h in (("q", hq), ("k", hk), ("v", hv), ("slot", hslot), ("ctx", hctx), ("bt", hbt)):
                S[name].copy_(h, non_blocking=True)
        ev_in[i].record(h2d)
        comp.wait_event(ev_in[i])
        comp.wait_event(ev_out[i])            # step k-2's output has been read back
        pkv.pkv_store_kvcache(S["k"], S["v"], c["kc"], c["vc"], S["slot"])
        pkv.pkv_decode(S["q"], c["kc"], c["vc"], S["bt"], S["ctx"], W.MAX_MODEL_LEN, W.SCALE, c["ws"],
                       out=S["out"])
        ev_done[i].record(comp)
        d2h.wait_event(ev_done[i])
        with torch.cuda.stream(d2h):
            hout[i].copy_(S["out"], non_blocking=True)
        ev_out[i].record(d2h)

    for k in range(max(3, args.warmup)):
        step(k)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(comp)
    h2d.wait_event(a)
    d2h.wait_event(a)
    for k in range(args.steps):
        step(k)
    comp.wait_stream(d2h)
    b.record(comp)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms = max_over_ranks(a.elapsed_time(b), world, dev) / args.steps
    if not torch.equal(hout[(args.steps - 1) % 2], c["out"].cpu()):
        raise RuntimeError("end-to-end output differs from the device-resident step")
    h2d_bytes = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hslot, hctx, hbt))
    return {"value": round(job_throughput(c["kv_bytes"], world, ms) / 1e9, 1), "unit": UNIT, "ms_per_step": round(ms, 5),
            "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": hout[0].numel() * hout[0].element_size(),
            "pipelining": "inputs and outputs double-buffered; copies on their own streams overlap the previous "
                          "step's kernels"}


def _prefill_flops(seqs):
    tot = 0
    for s in seqs:
        lq, lk = s.num_scheduled_tokens, s.num_cached_tokens + s.num_scheduled_tokens
        # sum over query rows of (position + 1) live keys
        tot += lq * (lk - lq) + lq * (lq + 1) // 2
    return 4 * W.HEAD_DIM * W.HQ * tot


def run_prefill(pkv, args, dev, bf16_peak, dtype=torch.bfloat16):
    f16 = dtype == torch.float16
    prefill = pkv.pkv_prefill_varlen_f16 if f16 else pkv.pkv_prefill_varlen
    flush = _make_flush(dev)
    res = {}
    iters = max(3, min(args.steps, 20))
    # calls of one workload run in order on one pool (chunked prompts continue
    # from the keys the previous calls stored)
    for name, wl in (("varlen_prefill_64p_len100-1024", W.varlen_prefill()),
                     ("prefix_prefill_128s_prefix1024_suffix64-512", W.prefix_prefill()),
                     ("chunked_prefill_16p_len4096-12288_budget5000", W.chunked_prefill())):
        gen = W.make_generator(wl.seed, dev)
        shape = (wl.num_blocks, W.BLOCK_SIZE, W.HKV, W.HEAD_DIM)
        kc, vc = W.normal(shape, gen, dev, dtype), W.normal(shape, gen, dev, dtype)
        calls = []
        for seqs in wl.seqs:
            T = sum(s.num_scheduled_tokens for s in seqs)
            _, q, k, v = W.fused_qkv(T, gen, dev, dtype=dtype)
            m = pkv.metadata.prepare_prefill(seqs, W.BLOCK_SIZE, force_block_tables=True)
            calls.append(dict(q=q, k=k, v=v, m=m, T=T, flops=_prefill_flops(seqs),
                              slot=torch.from_numpy(m["slot_mapping"]).to(dev),
                              cq=torch.from_numpy(m["cu_seqlens_q"]).to(dev),
                              ck=torch.from_numpy(m["cu_seqlens_k"]).to(dev),
                              bt=torch.from_numpy(m["block_tables"]).to(dev),
                              # the step's tile plan, built on the host with its metadata (untimed)
                              plan=pkv.pkv_prefill_plan(m["cu_seqlens_q"], m["cu_seqlens_k"], dev)))
        for it in range(iters + 3):
            _prequeue(0.5 * len(calls) + 1.0)  # host work per call below is ~0.1-0.25 ms
            for cl in calls:
                _flush_l2(flush)
                e0, e1, e2, e3, e4 = (torch.cuda.Event(enable_timing=True) for _ in range(5))
                e0.record()
                pkv.pkv_store_kvcache(cl["k"], cl["v"], kc, vc, cl["slot"])
                e1.record()
                prefill(cl["q"], cl["cq"], cl["ck"], cl["m"]["max_seqlen_q"], cl["m"]["max_seqlen_k"],
                        W.SCALE, k_cache=kc, v_cache=vc, block_tables=cl["bt"], plan=cl["plan"])
                e2.record()
                _flush_l2(flush)
                e3.record()
                prefill(cl["q"], cl["cq"], cl["ck"], cl["m"]["max_seqlen_q"], cl["m"]["max_seqlen_k"],
                        W.SCALE, k_cache=kc, v_cache=vc, block_tables=cl["bt"])
                e4.record()
                if it >= 3:
                    cl.setdefault("ev", []).append((e0, e1, e2, e3, e4))
        torch.cuda.synchronize()
        flops = sum(cl["flops"] for cl in calls)
        # which kernel ran each planned call; the workload's roofline names the
        # one that did most of its FLOPs, its traffic is that kernel's capture
        by_kernel = {}
        for cl in calls:
            kname = _prefill_kernel(cl["plan"].numel(), cl["m"]["max_seqlen_k"])
            by_kernel[kname] = by_kernel.get(kname, 0) + cl["flops"]
        kname, kfile = max(by_kernel, key=by_kernel.get)
        kernels = {k[0]: round(v / flops, 3) for k, v in by_kernel.items()}
        t_pre = sum(ev[1].elapsed_time(ev[2]) for cl in calls for ev in cl["ev"]) / iters
        t_noplan = sum(ev[3].elapsed_time(ev[4]) for cl in calls for ev in cl["ev"]) / iters
        t_st = sum(ev[0].elapsed_time(ev[1]) for cl in calls for ev in cl["ev"]) / iters
        store_bytes = sum(4 * int((cl["m"]["slot_mapping"] >= 0).sum()) * W.HKV * W.HEAD_DIM * 2 for cl in calls)
        tf = flops / (t_pre * 1e-3) / 1e12
        res[name] = {"calls": len(calls), "tokens": sum(cl["T"] for cl in calls), "gflop": round(flops / 1e9, 2),
                     "prefill_ms": round(t_pre, 4), "tflops": round(tf, 1),
                     "plan": "host tile plan per call (pkv_prefill_plan), built with the metadata, untimed",
                     "no_plan": {"prefill_ms": round(t_noplan, 4),
                                 "tflops": round(flops / (t_noplan * 1e-3) / 1e12, 1)},
                     "kernels_by_flop_share": kernels,
                     "roofline": {"kernel": kname, "bound": "tensor", "achieved": round(tf, 1),
                                  "peak": bf16_peak, "unit": "TFLOP/s", "frac": round(tf / bf16_peak, 4),
                                  "peak_source": ("measured bf16 dense (cuBLAS burst) x nominal fp16/bf16 ratio 1"
                                                  if f16 else "measured bf16 dense (cuBLAS burst)"),
                                  "traffic": None if f16 else _traffic(kfile, flops, case=name),
                                  "traffic_note": "ncu DRAM bytes of one planned launch: "
                                                  + str(_traffic_launch(kfile, name))},
                     "store_ms": round(t_st, 4), "store_gbs": round(store_bytes / (t_st * 1e-3) / 1e9, 1),
                     "l2": "256 MB buffer written, then another 256 MB read, between launches",
                     "queue": "launches queued behind a device-side sleep, so the events time the kernels, "
                              "not host launch latency"}
    assert pkv.pkv_device_error() == 0
    return res


def run_tiny(pkv, args, dev):
    """The 4-sequence decode step (contexts 37/256/300/511): latency in us of
    store + decode, eager launches and one graph replay; also the fused
    store + decode launch (pkv_store_decode) replayed in a graph."""
    wl = W.tiny_decode()
    gen = W.make_generator(wl.seed, dev)
    shape = (wl.num_blocks, W.BLOCK_SIZE, W.HKV, W.HEAD_DIM)
    kc, vc = W.normal(shape, gen, dev), W.normal(shape, gen, dev)
    B = len(wl.seqs)
    _, q, k, v = W.fused_qkv(B, gen, dev)
    m = pkv.metadata.prepare_decode(wl.seqs, W.BLOCK_SIZE)
    slot, ctx = torch.from_numpy(m["slot_mapping"]).to(dev), torch.from_numpy(m["context_lens"]).to(dev)
    bt = torch.from_numpy(m["block_tables"]).to(dev)
    ws = pkv.decode_workspace(B, W.MAX_MODEL_LEN, dev)
    out = torch.empty(B, W.HQ, W.HEAD_DIM, dtype=torch.bfloat16, device=dev)
    reps = max(10, min(args.steps, 200))

    def timed(fn, n):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record()
        for _ in range(n):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e3 / n

    def graph_of(fn):
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            fn()
        torch.cuda.current_stream().wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        return g

    def step():
        pkv.pkv_store_kvcache(k, v, kc, vc, slot)
        pkv.pkv_decode(q, kc, vc, bt, ctx, W.MAX_MODEL_LEN, W.SCALE, ws, out=out)

    def fused_step():
        pkv.pkv_store_decode(q, k, v, slot, kc, vc, bt, ctx, W.MAX_MODEL_LEN, W.SCALE, ws, out=out)

    for _ in range(args.warmup):
        step()
    eager_us = timed(step, reps)
    g = graph_of(step)
    for _ in range(args.warmup):
        g.replay()
    graph_us = timed(g.replay, reps)
    gf = graph_of(fused_step)
    for _ in range(args.warmup):
        gf.replay()
    fused_us = timed(gf.replay, reps)
    if pkv.pkv_device_error():
        raise RuntimeError("device error word set by the tiny decode")
    return {"workload": "tiny_decode_b4_ctx37/256/300/511: store 4 tokens + decode", "eager_us_per_step":
            round(eager_us, 2), "graph_us_per_step": round(graph_us, 2),
            "fused_graph_us_per_step": round(fused_us, 2), "steps": reps,
            "note": "latency-bound (4.5 MB of K/V); back-to-back steps, CUDA events; fused = pkv_store_decode, "
                    "one launch"}


def run_padded_graph(pkv, args, dev, hbm_peak):
    """200 live sequences decoded through a graph captured for 256 rows
    (store + decode), refreshed before every replay as the pages' run_model
    does: slot_mapping.fill_(-1), context_lens.zero_(), live part overwritten."""
    wl = W.padded_decode()
    B, G = len(wl.seqs), wl.graph_batch
    width = W.MAX_MODEL_LEN // W.BLOCK_SIZE
    gen = W.make_generator(wl.seed, dev)
    shape = (wl.num_blocks, W.BLOCK_SIZE, W.HKV, W.HEAD_DIM)
    kc, vc = W.normal(shape, gen, dev), W.normal(shape, gen, dev)
    meta = pkv.metadata.prepare_decode(wl.seqs, W.BLOCK_SIZE)
    _, q_new, k_new, v_new = W.fused_qkv(B, gen, dev)
    _, q, k, v = W.fused_qkv(G, gen, dev)
    slot = torch.full((G,), -1, dtype=torch.int32, device=dev)
    ctx = torch.zeros(G, dtype=torch.int32, device=dev)
    bt = torch.zeros(G, width, dtype=torch.int32, device=dev)
    out = torch.empty(G, W.HQ, W.HEAD_DIM, dtype=torch.bfloat16, device=dev)
    ws = pkv.decode_workspace(G, W.MAX_MODEL_LEN, dev)
    new_slot, new_ctx = torch.from_numpy(meta["slot_mapping"]).to(dev), torch.from_numpy(meta["context_lens"]).to(dev)
    new_bt = torch.from_numpy(meta["block_tables"]).to(dev)
    w = new_bt.shape[1]

    def refresh():
        slot.fill_(-1)
        ctx.zero_()
        bt[:B, :w] = new_bt
        slot[:B] = new_slot
        ctx[:B] = new_ctx
        q[:B], k[:B], v[:B] = q_new, k_new, v_new

    def step():
        pkv.pkv_store_kvcache(k, v, kc, vc, slot)
        pkv.pkv_decode(q, kc, vc, bt, ctx, W.MAX_MODEL_LEN, W.SCALE, ws, out=out)

    refresh()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    steps = max(3, min(args.steps, 100))
    evs = []
    for it in range(args.warmup + steps):
        refresh()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        if it >= args.warmup:
            evs.append((e0, e1))
    torch.cuda.synchronize()
    if pkv.pkv_device_error():
        raise RuntimeError("device error word set by the padded graph replay")
    ms = sum(a.elapsed_time(b) for a, b in evs) / len(evs)
    live_kv = int(meta["context_lens"].astype(np.int64).sum()) * W.HKV * W.HEAD_DIM * 2 * 2
    gbs = live_kv / (ms * 1e-3) / 1e9
    return {"workload": wl.name, "live_seqs": B, "graph_rows": G, "ms_per_replay": round(ms, 5),
            "live_kv_gbs": round(gbs, 1), "frac_of_hbm": round(gbs / hbm_peak, 4),
            "note": "replay time of store + decode only; the buffer refresh runs outside the events",
            "l2": "inputs larger than L2 (1.9 GB of live K/V per replay)"}


def run_f16(pkv, args, dev, hbm_peak, bf16_peak):
    """The fp16 entry points on the same workloads: decode (store + decode of
    the 256-sequence batch, kernel time by CUDA events) and both prefill cases."""
    c = decode_case(pkv, dev, dtype=torch.float16)
    stream = torch.cuda.current_stream()
    steps = max(3, min(args.steps, 50))
    evs = []
    for it in range(args.warmup + steps):
        pkv.pkv_store_kvcache(c["k"], c["v"], c["kc"], c["vc"], c["slot"])
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        pkv.pkv_decode_f16(c["q"], c["kc"], c["vc"], c["bt"], c["ctx"], W.MAX_MODEL_LEN, W.SCALE, c["ws"],
                           out=c["out"])
        e1.record(stream)
        if it >= args.warmup:
            evs.append((e0, e1))
    torch.cuda.synchronize()
    dec_ms = sum(a.elapsed_time(b) for a, b in evs) / len(evs)
    ach = c["decode_alg_bytes"] / (dec_ms * 1e-3) / 1e9
    if pkv.pkv_device_error():
        raise RuntimeError("device error word set by the fp16 decode")
    res = {"decode": {"workload": "batched_decode_b256_ctx512-4096 (fp16)", "avg_launch_ms": round(dec_ms, 5),
                      "roofline": {"kernel": _decode_kernel(c["B"]) + "<fp16>", "bound": "hbm", "achieved": round(ach, 1),
                                   "peak": hbm_peak, "unit": "GB/s", "frac": round(ach / hbm_peak, 4),
                                   "traffic": None}}}
    del c
    if not args.no_prefill:
        res["prefill"] = run_prefill(pkv, args, dev, bf16_peak, dtype=torch.float16)
    return res


def run_sweep(pkv, args, dev, hbm_peak):
    """28 layers x (store 512 tokens + decode 512 sequences), one CUDA graph."""
    wl = W.sweep_decode()
    L, B = wl.num_layers, len(wl.seqs)
    gen = W.make_generator(wl.seed, dev)
    kv = W.normal_bf16((2, L, wl.num_blocks, W.BLOCK_SIZE, W.HKV, W.HEAD_DIM), gen, dev)
    qkv = [W.fused_qkv(B, gen, dev) for _ in range(L)]
    meta = pkv.metadata.prepare_decode(wl.seqs, W.BLOCK_SIZE, table_width=W.MAX_MODEL_LEN // W.BLOCK_SIZE)
    slot = torch.from_numpy(meta["slot_mapping"]).to(dev)
    ctx = torch.from_numpy(meta["context_lens"]).to(dev)
    bt = torch.from_numpy(meta["block_tables"]).to(dev)
    ws = pkv.decode_workspace(B, W.MAX_MODEL_LEN, dev)
    outs = torch.empty(L, B, W.HQ, W.HEAD_DIM, dtype=torch.bfloat16, device=dev)

    def sweep():
        for l in range(L):
            _, q, k, v = qkv[l]
            pkv.pkv_store_kvcache(k, v, kv[0, l], kv[1, l], slot)
            pkv.pkv_decode(q, kv[0, l], kv[1, l], bt, ctx, W.MAX_MODEL_LEN, W.SCALE, ws, out=outs[l])

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        sweep()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        sweep()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    reps = max(3, min(args.steps, 20))
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / reps

    # the same sweep with the store fused into each decode launch (28 launches)
    def sweep_fused():
        for l in range(L):
            _, q, k, v = qkv[l]
            pkv.pkv_store_decode(q, k, v, slot, kv[0, l], kv[1, l], bt, ctx, W.MAX_MODEL_LEN, W.SCALE, ws,
                                 out=outs[l])

    with torch.cuda.stream(s):
        sweep_fused()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2):
        sweep_fused()
    for _ in range(3):
        g2.replay()
    torch.cuda.synchronize()
    a.record()
    for _ in range(reps):
        g2.replay()
    b.record()
    torch.cuda.synchronize()
    ms_fused = a.elapsed_time(b) / reps
    kv_bytes = L * int(meta["context_lens"].astype(np.int64).sum()) * W.HKV * W.HEAD_DIM * 4
    gbs = kv_bytes / (ms * 1e-3) / 1e9
    assert pkv.pkv_device_error() == 0
    del kv, g, g2
    torch.cuda.empty_cache()
    return {"workload": "decode_sweep_28l_b512_ctx_geometric800: 28 x (store 512 tokens + decode), one CUDA graph",
            "num_blocks": wl.num_blocks, "cache_gb": round(2 * L * wl.num_blocks * 256 * 8 * 128 * 2 / 1e9, 1),
            "sum_context_lens": int(meta["context_lens"].sum()), "ms_per_sweep": round(ms, 4),
            "kv_gbs": round(gbs, 1), "frac_of_hbm": round(gbs / hbm_peak, 4), "replays": reps,
            "gpu_launches_per_sweep": 2 * L,
            "fused_store_decode": {"ms_per_sweep": round(ms_fused, 4),
                                   "kv_gbs": round(kv_bytes / (ms_fused * 1e-3) / 1e9, 1),
                                   "frac_of_hbm": round(kv_bytes / (ms_fused * 1e-3) / 1e9 / hbm_peak, 4),
                                   "gpu_launches_per_sweep": L}}


def ncu_case(kind):
    """Small single-kernel cases for ncu captures (a few launches, a few GB)."""
    import paged_kv_cache_kvh_gb300 as pkv
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if kind == "decode":
        wl = W.batched_decode()
        seqs = wl.seqs[:64]
        used = sorted({b for s in seqs for b in s.block_table})
        remap = {b: i for i, b in enumerate(used)}
        seqs = [W.SeqSpec(s.num_tokens, [remap[b] for b in s.block_table]) for s in seqs]
        gen = W.make_generator(2, dev)
        shape = (len(used), W.BLOCK_SIZE, W.HKV, W.HEAD_DIM)
        kc, vc = W.normal_bf16(shape, gen, dev), W.normal_bf16(shape, gen, dev)
        _, q, k, v = W.fused_qkv(len(seqs), gen, dev)
        m = pkv.metadata.prepare_decode(seqs, W.BLOCK_SIZE, table_width=16)
        ws = pkv.decode_workspace(len(seqs), W.MAX_MODEL_LEN, dev)
        bt, ctx = torch.from_numpy(m["block_tables"]).to(dev), torch.from_numpy(m["context_lens"]).to(dev)
        for _ in range(3):
            pkv.pkv_decode(q, kc, vc, bt, ctx, W.MAX_MODEL_LEN, W.SCALE, ws)
        units = int(m["context_lens"].astype(np.int64).sum()) * W.HKV * W.HEAD_DIM * 4
    elif kind in ("prefill", "prefill_prefix", "prefill_chunked", "prefill_chunked_plain"):
        # the workload's first call; for the chunked workload call 9, a full
        # 5000-token chunk continuing 5000 cached tokens (whatever values the
        # seeded pool holds stand in for the keys the earlier call stored)
        # (prefill_chunked_plain: the same call without a tile plan, one CTA per unit)
        wl = {"prefill": W.varlen_prefill, "prefill_prefix": W.prefix_prefill,
              "prefill_chunked": W.chunked_prefill, "prefill_chunked_plain": W.chunked_prefill}[kind]()
        seqs = wl.seqs[9 if kind.startswith("prefill_chunked") else 0]
        gen = W.make_generator(wl.seed, dev)
        shape = (wl.num_blocks, W.BLOCK_SIZE, W.HKV, W.HEAD_DIM)
        kc, vc = W.normal_bf16(shape, gen, dev), W.normal_bf16(shape, gen, dev)
        T = sum(s.num_scheduled_tokens for s in seqs)
        _, q, k, v = W.fused_qkv(T, gen, dev)
        m = pkv.metadata.prepare_prefill(seqs, W.BLOCK_SIZE, force_block_tables=True)
        d = lambda a: torch.from_numpy(a).to(dev)  # noqa: E731
        pkv.pkv_store_kvcache(k, v, kc, vc, d(m["slot_mapping"]))
        plan = None if kind == "prefill_chunked_plain" else pkv.pkv_prefill_plan(m["cu_seqlens_q"],
                                                                                 m["cu_seqlens_k"], dev)
        for _ in range(3):
            pkv.pkv_prefill_varlen(q, d(m["cu_seqlens_q"]), d(m["cu_seqlens_k"]), m["max_seqlen_q"],
                                   m["max_seqlen_k"], W.SCALE, k_cache=kc, v_cache=vc, block_tables=d(m["block_tables"]),
                                   plan=plan)
        units = _prefill_flops(seqs)
    elif kind == "sweep":
        # the 28-layer sweep, one eager pass (store + decode per layer): 56 launches
        # on a 54 GB cache, for a one-metric launch list only
        wl = W.sweep_decode()
        L, B = wl.num_layers, len(wl.seqs)
        gen = W.make_generator(wl.seed, dev)
        kv = W.normal_bf16((2, L, wl.num_blocks, W.BLOCK_SIZE, W.HKV, W.HEAD_DIM), gen, dev)
        m = pkv.metadata.prepare_decode(wl.seqs, W.BLOCK_SIZE, table_width=W.MAX_MODEL_LEN // W.BLOCK_SIZE)
        d = lambda a: torch.from_numpy(a).to(dev)  # noqa: E731
        slot, ctx, bt = d(m["slot_mapping"]), d(m["context_lens"]), d(m["block_tables"])
        ws = pkv.decode_workspace(B, W.MAX_MODEL_LEN, dev)
        qkv = [W.fused_qkv(B, gen, dev) for _ in range(L)]
        torch.cuda.synchronize()
        for l in range(L):
            _, q, k, v = qkv[l]
            pkv.pkv_store_kvcache(k, v, kv[0, l], kv[1, l], slot)
            pkv.pkv_decode(q, kv[0, l], kv[1, l], bt, ctx, W.MAX_MODEL_LEN, W.SCALE, ws)
        units = L * int(m["context_lens"].astype(np.int64).sum()) * W.HKV * W.HEAD_DIM * 4
    elif kind == "store":
        gen = W.make_generator(3, dev)
        N = 16384
        kc = W.normal_bf16((160, W.BLOCK_SIZE, W.HKV, W.HEAD_DIM), gen, dev)
        vc = W.normal_bf16((160, W.BLOCK_SIZE, W.HKV, W.HEAD_DIM), gen, dev)
        _, q, k, v = W.fused_qkv(N, gen, dev)
        slot = torch.from_numpy(np.random.default_rng(3).permutation(160 * 256)[:N].astype(np.int32)).to(dev)
        for _ in range(3):
            pkv.pkv_store_kvcache(k, v, kc, vc, slot)
        units = N * W.HKV * W.HEAD_DIM * 8
    else:
        raise SystemExit(f"unknown ncu case {kind}")
    torch.cuda.synchronize()
    assert pkv.pkv_device_error() == 0
    print(json.dumps({"ncu_case": kind, "units": units}))


# ---------------------------------------------------------------------------
# oracle (CPU) arm
# ---------------------------------------------------------------------------

def _oracle_sample(num_sample, seed=2):
    """The first num_sample sequences of the batched-decode workload, their
    blocks generated on the host (compact pool), for the oracle."""
    import oracle
    wl = W.batched_decode(seed=seed)
    seqs = wl.seqs[:num_sample]
    used = sorted({b for s in seqs for b in s.block_table})
    remap = {b: i for i, b in enumerate(used)}
    gen = W.make_generator(seed, "cpu")
    shape = (len(used), W.BLOCK_SIZE, W.HKV, W.HEAD_DIM)
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    kc, vc = bits(W.normal_bf16(shape, gen, "cpu")), bits(W.normal_bf16(shape, gen, "cpu"))
    _, q, k, v = W.fused_qkv(num_sample, gen, "cpu")
    osq = [oracle.SeqState(s.num_tokens, [remap[b] for b in s.block_table]) for s in seqs]
    m = oracle.prepare_decode(osq, W.BLOCK_SIZE)
    kv_bytes = int(m["context_lens"].astype(np.int64).sum()) * W.HKV * W.HEAD_DIM * 4
    return dict(q=bits(q), k=bits(k), v=bits(v), kc=kc, vc=vc, m=m, kv_bytes=kv_bytes, n=num_sample)


def _oracle_step(orc, s):
    import oracle  # noqa: F401
    orc.store_kvcache(s["k"], s["v"], s["kc"].reshape(-1, W.HKV, W.HEAD_DIM), s["vc"].reshape(-1, W.HKV, W.HEAD_DIM),
                      s["m"]["slot_mapping"])
    orc.decode(s["q"], s["kc"], s["vc"], s["m"]["block_tables"], s["m"]["context_lens"], W.SCALE,
               num_kv_heads=W.HKV)


def _cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=5).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_baseline(c=None, budget_s=10.0, num_sample=16):
    import oracle
    orc = oracle.default()
    s = _oracle_sample(num_sample)
    t0 = time.perf_counter()
    reps = 0
    while True:
        _oracle_step(orc, s)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= 1000:
            break
    return {"value": round(s["kv_bytes"] * reps / el / 1e9, 4), "unit": UNIT, "cores": orc.num_threads(),
            "cpu_model": _cpu_model(), "kind": "oracle", "sample": f"store + decode of the first {num_sample} of the 256 sequences "
                                       f"(fp64 C oracle), repeated {reps}x over {el:.1f} s"}


def run_reference(args):
    import oracle
    orc = oracle.default()
    s = _oracle_sample(args.ref_sample)
    for _ in range(args.warmup):
        _oracle_step(orc, s)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_step(orc, s)
    el = time.perf_counter() - t0
    ms = el * 1e3 / args.steps
    val = round(s["kv_bytes"] / (ms * 1e-3) / 1e9, 4)
    return {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1) bf16, shuffled block tables)",
            "config": {"workload": "batched_decode_b256_ctx512-4096: store_kvcache(256 tokens) + GQA decode",
                       "sample_seqs": args.ref_sample},
            "cpu_baseline": {"value": val, "unit": UNIT, "kind": "oracle", "cores": orc.num_threads(),
                             "cpu_model": _cpu_model(),
                             "sample": f"each step: store + decode of the first {args.ref_sample} of the 256 "
                                       f"sequences with the fp64 C oracle"},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-sample", type=int, default=8)
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-f16", action="store_true", help="skip the fp16 entry points' timings")
    ap.add_argument("--ncu-case", choices=["decode", "prefill", "prefill_prefix", "prefill_chunked",
                                           "prefill_chunked_plain", "store", "sweep"])
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.ncu_case:
        ncu_case(args.ncu_case)
        return

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    try:
        res = run_ours(args, rank, world, dev)
        if rank == 0:
            print(json.dumps(res), flush=True)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
