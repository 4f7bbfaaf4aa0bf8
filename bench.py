"""Benchmark of the attention-sublayer hot path on GB300.

One step = one Qwen3-8B decode layer step (add-RMSNorm [256, 4096],
QK-Norm + RoPE of 256 new tokens, store_kvcache of their K/V, paged decode
attention for 256 sequences with contexts ~ U[1024, 8192]) followed by one
Qwen3-8B varlen prefill step (16 sequences of U[128, 4096] tokens: add-RMSNorm,
QK-Norm + RoPE, store_kvcache of every token, causal prefill attention).

Reported (one JSON line on rank 0):
  value      decode-step throughput in GB/s of algorithmic HBM bytes (the
             metric's first figure); inputs resident in HBM.
  prefill    prefill attention TFLOP/s over the causal pairs (second figure).
  roofline   the dominant kernel (paged decode attention) against the
             measured HBM copy peak; prefill against the bf16 tensor peak.
  e2e        the decode step through the C-ABI with pinned host inputs copied
             in and outputs copied back inside the timed region.
  cpu_baseline  the fp64 oracle on a bounded sample of the decode step.
L2 is flushed between timed steps, outside the events: 256 MB are written, then a
different 256 MB buffer is read, so the timed kernels find neither their inputs
nor dirty lines (whose write-back they would pay for) in L2.

--impl reference times the oracle alone (the CPU reference arm).
--gpus N under torchrun runs N independent replicas (the path needs no
exchange between GPUs), value = total bytes of all ranks / max time.
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "paged-attn decode HBM GB/s (% peak); prefill attn TFLOP/s, Qwen3-8B shape"
WORKLOAD = ("qwen3-8b attention sublayer step: decode layer B=256 ctx~U[1024,8192] "
            "(add-RMSNorm, QK-Norm+RoPE, store_kvcache, paged decode) + prefill layer "
            "16 seqs U[128,4096] (add-RMSNorm, QK-Norm+RoPE, store_kvcache, varlen causal "
            "prefill)")
SEQ_LEN = "ctx U[1024,8192]; prefill U[128,4096]"
SCALE = 128 ** -0.5


# DRAM bytes per algorithmic byte of the decode attention kernels, from an
# ncu capture of `bench.py --ncu-case decode` (reads + writes of
# decode_split_kernel and decode_merge_kernel over the algorithmic bytes),
# valid only for the kernel code it was taken on (the hash ignores comments
# and layout).
DECODE_TRAFFIC = {"ratio": 1.0036, "source_sha256_16": "5574a127e6991e65"}
# DRAM bytes (read + write) of one prefill-attention launch on the bench batch
# (33,109 tokens, Qwen3-8B heads): mean of the two launches of an ncu capture
# of `bench.py --ncu-case layer` (cold L2, as ncu runs each launch).
PREFILL_TRAFFIC = {"bytes": 1179100800, "source_sha256_16": "2e2f80d5fe096d24"}


def max_over_ranks(values, world: int, device=None):
    """Each timing's maximum over all ranks: the slowest replica sets the
    job's time.  With one rank the values come back unchanged."""
    values = [float(v) for v in values]
    if world <= 1:
        return values
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_throughput(units_per_rank: float, world: int, seconds: float) -> float:
    """Whole-job rate: the units every rank processed over the slowest
    rank's time (replicas each do the same work)."""
    return world * units_per_rank / seconds


def strip_comments(src: str) -> str:
    """C/CUDA source without its comments, whitespace runs collapsed (string
    and character literals kept as they are)."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash(name: str) -> str:
    """Hash of a kernel source's code: comments and layout do not count, so a
    traffic figure taken on the code stays valid across comment edits."""
    import hashlib
    path = os.path.join(ROOT, "paged_kv_attention_kvcache_gb300", "csrc", name)
    with open(path, encoding="utf-8") as f:
        return hashlib.sha256(strip_comments(f.read()).encode()).hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), \
            "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


class L2Flush:
    """Clears L2 between timed reps: writes a 256 MB buffer (evicting every
    input), then reads a second one, so that L2 is left holding clean lines
    only and the next timed kernel pays no write-back of the flush's data."""

    def __init__(self, dev_t, mb: int = 256):
        import torch
        n = mb * 1024 * 1024 // 4
        self.w = torch.empty(n, dtype=torch.float32, device=dev_t)
        self.r = torch.zeros(n, dtype=torch.float32, device=dev_t)

    def __call__(self):
        self.w.zero_()
        self.r.sum()


# ------------------------------------------------------- algorithmic bytes
def decode_step_bytes(step: wl.DecodeStep) -> dict:
    s = step.shape
    B = step.context_lens.size
    H, Q, D = s.hidden, s.q_size, s.kv_size
    ctx = step.context_lens.astype(np.int64)
    blocks = np.ceil(ctx / wl.BLOCK_SIZE).astype(np.int64)
    norm = B * H * 2 * 4 + H * 2
    qkn = B * (Q + D) * 2 * 2 + B * (8 + 128 * 4) + 2 * 128 * 2
    store = B * D * 2 * 4 + B * 4
    attn = int(ctx.sum()) * D * 2 * 2 + B * Q * 2 * 2 + int(blocks.sum()) * 4 + B * 4
    return dict(norm=norm, qknorm_rope=qkn, store=store, attn=attn,
                total=norm + qkn + store + attn)


def prefill_flops(lengths) -> float:
    L = np.asarray(lengths, dtype=np.float64)
    return float(4 * 128 * 32 * np.sum(L * (L + 1) / 2))


# ------------------------------------------------------------- clock probe
class ClockSampler:
    """nvidia-smi sampled every 20 ms in a reader thread; `window()` keeps
    the samples taken between mark_start() and mark_end(), `between(t0, t1)`
    those of any other interval."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index: int):
        import threading
        self.samples = []
        self.t0 = self.t1 = None
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        deadline = time.time() + 10
        while not self.samples and time.time() < deadline:
            time.sleep(0.02)

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        if self.proc is None or self.proc.poll() is not None:
            return
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()

    def summarize(self, lines):
        sm, smax, reasons = [], None, set()
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(self.NAMES, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}

    def between(self, t0, t1):
        return self.summarize([l for t, l in self.samples if t0 <= t <= t1])

    def window(self):
        if self.proc is None:
            return None
        inside = [l for t, l in self.samples if self.t0 is not None and self.t0 <= t <= self.t1]
        used = inside if inside else [l for _, l in self.samples[-3:]]
        out = self.summarize(used)
        if out is not None:
            out["in_window"] = bool(inside)
        return out


# ---------------------------------------------------------------- our arm
def run_ours(args, rank, world, local_rank):
    import torch
    import paged_kv_attention_kvcache_gb300 as nv

    torch.cuda.set_device(local_rank)
    dev_t = torch.device("cuda", local_rank)

    def dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(
            torch.bfloat16).to(dev_t)

    def i32(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev_t)

    def i64(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int64)).to(dev_t)

    t_gen = time.time()
    step = wl.config3()
    pre = wl.config4()
    gen_s = time.time() - t_gen
    s = step.shape
    B = step.context_lens.size
    H, Q, D = s.hidden, s.q_size, s.kv_size
    err = torch.zeros(1, dtype=torch.int32, device=dev_t)
    table = torch.empty(wl.MAX_POSITION, 128, dtype=torch.float32, device=dev_t)
    nv.nv_rope_cos_sin_cache(table, wl.ROPE_BASE)

    # ---- decode state
    kc, vc = dev(step.pool.k), dev(step.pool.v)
    d_x, d_r, d_g = dev(step.x), dev(step.residual), dev(step.gamma)
    d_y = torch.empty_like(d_x)
    d_qkv = dev(step.qkv)
    d_qn, d_kn = dev(step.q_norm_w), dev(step.k_norm_w)
    d_pos, d_slots = i64(step.positions), i32(step.slot_mapping)
    d_bt, d_ctx = i32(step.block_tables), i32(step.context_lens)
    d_o = torch.empty(B, s.hq, 128, dtype=torch.bfloat16, device=dev_t)
    ws_bytes = nv.nv_decode_attn_workspace_size(B, s.hq, s.hkv, 128, step.block_tables.shape[1],
                                                wl.BLOCK_SIZE, 0)
    ws = torch.empty(max(1, ws_bytes // 4), dtype=torch.float32, device=dev_t)
    decode_kernels = 2 if ws_bytes else 1

    def decode_views(qkv):
        return (qkv[:, :Q].view(B, s.hq, 128), qkv[:, Q:Q + D].view(B, s.hkv, 128),
                qkv[:, Q + D:].view(B, s.hkv, 128))

    dq, dk, dv = decode_views(d_qkv)

    def decode_attn():
        nv.nv_decode_attn_paged(dq, kc, vc, d_bt, d_ctx, d_o, SCALE, workspace=ws,
                                err_count=err)

    def decode_layer(x=d_x, r=d_r, y=d_y, q=dq, k=dk, v=dv, pos=d_pos, slots=d_slots,
                     bt=d_bt, ctx=d_ctx, o=d_o, ev=None):
        nv.nv_add_rmsnorm(x, r, d_g, y, r, eps=wl.RMS_EPS)
        nv.nv_qknorm_rope(q, k, d_qn, d_kn, table, pos, eps=wl.RMS_EPS, err_count=err)
        nv.nv_store_kvcache(k, v, kc, vc, slots, err)
        if ev:
            ev[0].record()
        nv.nv_decode_attn_paged(q, kc, vc, bt, ctx, o, SCALE, workspace=ws, err_count=err)
        if ev:
            ev[1].record()

    # ---- prefill state
    T = pre.qkv.shape[0]
    p_x, p_r, p_g = dev(pre.x), dev(pre.residual), dev(pre.gamma)
    p_y = torch.empty_like(p_x)
    p_qkv = dev(pre.qkv)
    p_qn, p_kn = dev(pre.q_norm_w), dev(pre.k_norm_w)
    p_pos, p_slots, p_cu = i64(pre.positions), i32(pre.slot_mapping), i32(pre.cu_seqlens)
    pkc = torch.zeros(pre.num_blocks, wl.BLOCK_SIZE, s.hkv, 128, dtype=torch.bfloat16,
                      device=dev_t)
    pvc = torch.zeros_like(pkc)
    p_o = torch.empty(T, s.hq, 128, dtype=torch.bfloat16, device=dev_t)
    pq, pk, pv = (p_qkv[:, :Q].view(T, s.hq, 128), p_qkv[:, Q:Q + D].view(T, s.hkv, 128),
                  p_qkv[:, Q + D:].view(T, s.hkv, 128))
    max_len = int(pre.lengths.max())
    p_sched = torch.zeros(1, dtype=torch.int32, device=dev_t)   # dynamic work counter

    def prefill_layer(ev=None):
        nv.nv_add_rmsnorm(p_x, p_r, p_g, p_y, p_r, eps=wl.RMS_EPS)
        nv.nv_qknorm_rope(pq, pk, p_qn, p_kn, table, p_pos, eps=wl.RMS_EPS, err_count=err)
        nv.nv_store_kvcache(pk, pv, pkc, pvc, p_slots, err)
        if ev:
            ev[0].record()
        nv.nv_prefill_attn_varlen(pq, pk, pv, p_o, p_cu, p_cu, max_len, max_len, SCALE,
                                  err_count=err, sched_counter=p_sched)
        if ev:
            ev[1].record()

    launches_per_step = (3 + decode_kernels) + 4
    flush = L2Flush(dev_t)

    def ev():
        return torch.cuda.Event(enable_timing=True)

    clocks = ClockSampler(local_rank)
    for _ in range(args.warmup):
        decode_layer()
        prefill_layer()
    torch.cuda.synchronize()

    # ---- timed region
    records = []
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    clocks.mark_start()
    t_wall = time.time()
    for _ in range(args.steps):
        flush()
        e = [ev() for _ in range(6)]
        e[0].record()
        decode_layer(ev=(e[1], e[2]))
        e[3].record()
        prefill_layer(ev=(e[4], e[5]))
        records.append(e)
    torch.cuda.synchronize()
    wall = time.time() - t_wall
    clocks.mark_end()
    if world > 1:
        dist.barrier()
    clk = clocks.window()

    # ---- clock block: the same step repeated for at least 1.2 s (L2 not
    # flushed), so that clock samples taken every 20 ms cover the work they
    # are quoted with: time x median SM clock gives cycles per step.
    mean_step_ms = statistics.mean(e[0].elapsed_time(e[3]) + e[3].elapsed_time(e[5])
                                   for e in records)
    n_blk = max(50, int(1.2e3 / max(0.1, mean_step_ms)))
    torch.cuda.synchronize()
    eb0, eb1 = ev(), ev()
    tb0 = time.time()
    eb0.record()
    for _ in range(n_blk):
        decode_layer()
        prefill_layer()
    eb1.record()
    torch.cuda.synchronize()
    tb1 = time.time()
    blk_ms = eb0.elapsed_time(eb1) / n_blk
    bclk = clocks.between(tb0, tb1)
    clocks.stop()
    clock_block = {"steps": n_blk, "seconds": round(tb1 - tb0, 3), "ms_per_step": blk_ms,
                   "l2": "not flushed"}
    if bclk:
        clock_block.update(sm_mhz_median=bclk["sm_mhz"], sm_max_mhz=bclk["sm_max_mhz"],
                           reasons=bclk["reasons"], samples=bclk["samples"],
                           kcycles_per_step=blk_ms * bclk["sm_mhz"])
    dec_ms = [e[0].elapsed_time(e[3]) for e in records]
    attn_ms = [e[1].elapsed_time(e[2]) for e in records]
    pre_ms = [e[3].elapsed_time(e[5]) for e in records]
    pattn_ms = [e[4].elapsed_time(e[5]) for e in records]
    step_ms = [a + b for a, b in zip(dec_ms, pre_ms)]
    assert int(err.item()) == 0, f"device error count {int(err.item())}"

    dec_time, tot_ms, pattn_sum = max_over_ranks(
        [sum(dec_ms) / 1e3, sum(step_ms), sum(pattn_ms)], world, dev_t)

    nbytes = decode_step_bytes(step)
    hbm, bf16, bf16_sus, peak_src = measured_peaks()
    value = job_throughput(nbytes["total"] * args.steps, world, dec_time) / 1e9
    attn_avg_s = statistics.mean(attn_ms) / 1e3
    attn_gbs = nbytes["attn"] / attn_avg_s / 1e9
    pflops = prefill_flops(pre.lengths)
    ptflops = pflops / (pattn_sum / args.steps / 1e3) / 1e12

    # ---- e2e: host buffers through the C-ABI, host<->device traffic inside the
    # timed region.  add-RMSNorm reads x and the residual straight from pinned
    # host memory and writes y and the new residual straight back (the ABI
    # takes device-addressable host pointers for tensors its kernels touch with
    # plain loads and stores); qkv and the metadata go over in one packed
    # copy (the rotation works in place, and the host inputs must stay as they
    # are for the next step); the decode kernel writes o to pinned host memory.
    # One stream, in the layer's order.
    MB = step.block_tables.shape[1]
    in_specs = [("qkv", step.qkv.view(np.int16), torch.bfloat16),
                ("pos", step.positions, torch.int64),
                ("slots", step.slot_mapping, torch.int32),
                ("bt", step.block_tables, torch.int32),
                ("ctx", step.context_lens, torch.int32)]
    offs, off = {}, 0
    for name, arr, _ in in_specs:
        offs[name] = off
        off += (arr.nbytes + 255) // 256 * 256
    host_in = torch.zeros(off, dtype=torch.uint8).pin_memory()
    for name, arr, _ in in_specs:
        host_in[offs[name]:offs[name] + arr.nbytes].copy_(
            torch.from_numpy(np.ascontiguousarray(arr).view(np.uint8).reshape(-1)))
    dev_in = torch.empty(off, dtype=torch.uint8, device=dev_t)
    dv = {name: dev_in[offs[name]:offs[name] + arr.nbytes].view(dt).view(arr.shape)
          for name, arr, dt in in_specs}
    host_x = torch.from_numpy(step.x.view(np.int16)).view(torch.bfloat16).pin_memory()
    host_r = torch.from_numpy(step.residual.view(np.int16)).view(torch.bfloat16).pin_memory()
    host_y = torch.empty(B, H, dtype=torch.bfloat16).pin_memory()
    host_rout = torch.empty(B, H, dtype=torch.bfloat16).pin_memory()
    host_o = torch.empty(B, s.hq, 128, dtype=torch.bfloat16).pin_memory()
    h2d = sum(arr.nbytes for _, arr, _ in in_specs) + 2 * host_x.numel() * 2
    d2h = (host_y.numel() + host_rout.numel() + host_o.numel()) * 2
    q2, k2, v2 = decode_views(dv["qkv"])
    e2e_ms = []
    for i in range(args.warmup + args.steps):
        flush()
        e0, e1 = ev(), ev()
        e0.record()
        nv.nv_add_rmsnorm(host_x, host_r, d_g, host_y, host_rout, eps=wl.RMS_EPS)
        dev_in.copy_(host_in, non_blocking=True)
        nv.nv_qknorm_rope(q2, k2, d_qn, d_kn, table, dv["pos"], eps=wl.RMS_EPS, err_count=err)
        nv.nv_store_kvcache(k2, v2, kc, vc, dv["slots"], err)
        nv.nv_decode_attn_paged(q2, kc, vc, dv["bt"], dv["ctx"], host_o, SCALE, workspace=ws,
                                err_count=err)
        e1.record()
        torch.cuda.synchronize()
        if i >= args.warmup:
            e2e_ms.append(e0.elapsed_time(e1))
    e2e_s = max_over_ranks([statistics.mean(e2e_ms) / 1e3], world, dev_t)[0]
    e2e_val = job_throughput(nbytes["total"], world, e2e_s) / 1e9

    graph_info = graph_decode_overhead(dev_t)
    decode_sets_out = decode_sets(dev_t, measured_peaks()[0])
    prefix_prefill = prefill_prefix_config(dev_t)

    # ---- QK-Norm + RoPE + store on the prefill batch: two kernels vs one pass
    def time_us(fn, reps=20):
        for _ in range(3):
            fn()
        e0, e1 = ev(), ev()
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / reps

    def pair():
        nv.nv_qknorm_rope(pq, pk, p_qn, p_kn, table, p_pos, eps=wl.RMS_EPS, err_count=err)
        nv.nv_store_kvcache(pk, pv, pkc, pvc, p_slots, err)

    def fused():
        nv.nv_qknorm_rope_store(pq, pk, pv, p_qn, p_kn, table, p_pos, pkc, pvc, p_slots,
                                eps=wl.RMS_EPS, write_k=True, err_count=err)

    pair_us, fused_us = time_us(pair), time_us(fused)
    # q and k read and written by the rotation, k and v read and written by the store;
    # the fused pass reads q, k, v once and writes q, k and both cache rows.
    pair_bytes = T * (2 * (Q + D) + 4 * D) * 2
    fused_bytes = T * ((Q + 2 * D) + (Q + D) + 2 * D) * 2
    rope_store = {"tokens": T, "write_k": True, "pair_us": pair_us, "fused_us": fused_us,
                  "pair_bytes": pair_bytes, "fused_bytes": fused_bytes,
                  "fused_gbs": fused_bytes / (fused_us * 1e-6) / 1e9,
                  "pair_gbs": pair_bytes / (pair_us * 1e-6) / 1e9}
    hbm_peak = measured_peaks()[0]
    rope_store["fused_frac"] = rope_store["fused_gbs"] / hbm_peak
    rope_store["pair_frac"] = rope_store["pair_gbs"] / hbm_peak
    assert int(err.item()) == 0, f"device error count {int(err.item())}"

    # ---- the MLP's SiluAndMul on the prefill batch (Qwen3-8B intermediate 12288)
    inter = 12288
    gate_up = torch.empty(T, 2 * inter, dtype=torch.bfloat16, device=dev_t).normal_()
    act = torch.empty(T, inter, dtype=torch.bfloat16, device=dev_t)
    swiglu_us = time_us(lambda: nv.nv_silu_and_mul(gate_up, act))
    swiglu_bytes = T * 3 * inter * 2
    swiglu = {"tokens": T, "intermediate": inter, "us": swiglu_us, "bytes": swiglu_bytes,
              "gbs": swiglu_bytes / (swiglu_us * 1e-6) / 1e9}
    swiglu["frac"] = swiglu["gbs"] / hbm_peak
    del gate_up, act

    return dict(
        graph=graph_info, rope_store=rope_store, swiglu=swiglu, decode_sets=decode_sets_out,
        prefix_prefill=prefix_prefill,
        value=value, ms_per_step=tot_ms / args.steps, dec_ms=statistics.mean(dec_ms),
        pre_ms=statistics.mean(pre_ms), attn_ms=statistics.mean(attn_ms),
        attn_gbs=attn_gbs, ptflops=ptflops, pattn_ms=pattn_sum / args.steps, clocks=clk,
        clock_block=clock_block,
        hbm=hbm, bf16=bf16, bf16_sus=bf16_sus, peak_src=peak_src, nbytes=nbytes,
        launches=launches_per_step * args.steps, e2e=e2e_val, h2d=h2d, d2h=d2h, wall=wall,
        gen_s=gen_s, step=step, pre=pre, ws_bytes=ws_bytes, T=T)


# ------------------------------------------------------ the other decode sets
def store_decode_bytes(step: wl.DecodeStep) -> dict:
    """Algorithmic bytes of a decode step without the norms: store_kvcache of
    the new token's K/V (read k, v; write both cache rows; slot) and paged
    decode attention (K/V read once per kv head, q, o, block table, context)."""
    s = step.shape
    B = step.context_lens.size
    Q, D = s.q_size, s.kv_size
    ctx = step.context_lens.astype(np.int64)
    blocks = np.ceil(ctx / wl.BLOCK_SIZE).astype(np.int64)
    store = B * D * 2 * 4 + B * 4
    attn = int(ctx.sum()) * D * 2 * 2 + B * Q * 2 * 2 + int(blocks.sum()) * 4 + B * 4
    return dict(store=store, attn=attn, total=store + attn)


def decode_sets(dev_t, hbm_peak: float, reps: int = 20):
    """The two other decode workloads, each timed (L2 flushed before each rep,
    median of `reps` event-timed reps):
      Qwen3-0.6B heads, B=64, ctx U[512, 4096]: the whole step as the pages run
        it -- store_kvcache of each sequence's new token, then paged decode --
        and the attention call alone;
      Qwen3-8B heads, B=32, ctx log-U[4096, 40960], 1% outlier K rows: paged
        decode with the automatic split and with forced 1024-key splits."""
    import torch
    import paged_kv_attention_kvcache_gb300 as nv
    flush = L2Flush(dev_t)

    def dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(
            torch.bfloat16).to(dev_t)

    def timed(fn):
        times = []
        for i in range(reps + 3):
            flush()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            if i >= 3:
                times.append(e0.elapsed_time(e1) / 1e3)
        return statistics.median(times)

    def entry(nbytes, t, B, what):
        gbs = nbytes / t / 1e9
        return {"what": what, "bytes": nbytes, "ms": t * 1e3, "gbs": gbs,
                "frac": gbs / hbm_peak, "tokens_per_s": B / t}

    out = {}
    # ---- Qwen3-0.6B heads, B = 64: store then decode
    step = wl.config2()
    s = step.shape
    B, Q, D = step.context_lens.size, s.q_size, s.kv_size
    qkv = dev(step.qkv)
    q = qkv[:, :Q].view(B, s.hq, 128)
    k = qkv[:, Q:Q + D].view(B, s.hkv, 128)
    v = qkv[:, Q + D:].view(B, s.hkv, 128)
    kc, vc = dev(step.pool.k), dev(step.pool.v)
    bt = torch.from_numpy(step.block_tables).to(dev_t)
    cl = torch.from_numpy(step.context_lens).to(dev_t)
    slots = torch.from_numpy(step.slot_mapping).to(dev_t)
    o = torch.empty(B, s.hq, 128, dtype=torch.bfloat16, device=dev_t)
    wsb = nv.nv_decode_attn_workspace_size(B, s.hq, s.hkv, 128, bt.shape[1], wl.BLOCK_SIZE, 0)
    ws = torch.empty(max(1, wsb // 4), dtype=torch.float32, device=dev_t)
    nb = store_decode_bytes(step)

    def attn():
        nv.nv_decode_attn_paged(q, kc, vc, bt, cl, o, SCALE, workspace=ws)

    def full_step():
        nv.nv_store_kvcache(k, v, kc, vc, slots)
        attn()

    out["b64_ctx512_4096_qwen3_06b_step"] = entry(
        nb["total"], timed(full_step), B, "store_kvcache of 64 new tokens + paged decode")
    out["b64_ctx512_4096_qwen3_06b_attn"] = entry(nb["attn"], timed(attn), B,
                                                   "paged decode alone")
    out["b64_ctx512_4096_qwen3_06b_attn"]["kv_bytes"] = nb["attn"]
    del kc, vc, qkv
    # ---- Qwen3-8B heads, B = 32, long contexts
    step = wl.config5()
    s = step.shape
    B = step.context_lens.size
    q = dev(step.qkv[:, :s.q_size]).view(B, s.hq, 128)
    kc, vc = dev(step.pool.k), dev(step.pool.v)
    bt = torch.from_numpy(step.block_tables).to(dev_t)
    cl = torch.from_numpy(step.context_lens).to(dev_t)
    o = torch.empty(B, s.hq, 128, dtype=torch.bfloat16, device=dev_t)
    nbytes = store_decode_bytes(step)["attn"]
    for split in (0, 1024):
        wsb = nv.nv_decode_attn_workspace_size(B, s.hq, s.hkv, 128, bt.shape[1],
                                               wl.BLOCK_SIZE, split)
        ws = torch.empty(max(1, wsb // 4), dtype=torch.float32, device=dev_t)
        t = timed(lambda: nv.nv_decode_attn_paged(q, kc, vc, bt, cl, o, SCALE, workspace=ws,
                                                  kv_split_tokens=split))
        out[f"b32_ctx4096_40960_qwen3_8b_split{split or 'auto'}"] = entry(
            nbytes, t, B, f"paged decode, {'automatic' if not split else '1024-key'} split")
    del kc, vc, flush
    return out


# ------------------------------------ prefill over the paged cache (prefix hit)
def prefill_prefix_config(dev_t, reps: int = 20):
    """Prefill over the paged cache on the prefix-hit workload (Qwen3-8B heads,
    16 sequences, cached prefixes of 256..4096 tokens, 128..1024 new ones):
    nv_prefill_attn_paged, and nv_prefill_attn_varlen over the same keys
    gathered into contiguous rows.  FLOPs count the causal pairs only,
    4*d*Hq*sum(L*P + L*(L+1)/2).  L2 flushed before each rep; median of `reps`
    event-timed launches."""
    import torch
    import paged_kv_attention_kvcache_gb300 as nv
    pre = wl.config_prefix()
    s = pre.shape
    L = pre.new.astype(np.float64)
    P = pre.prefix.astype(np.float64)
    flops = float((4 * 128 * s.hq * (L * P + L * (L + 1) / 2)).sum())

    def dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(
            torch.bfloat16).to(dev_t)

    def dev_i32(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev_t)

    flush = L2Flush(dev_t)
    q, kc, vc = dev(pre.q), dev(pre.pool.k), dev(pre.pool.v)
    kk, vv = wl.gather_paged(pre.pool, pre.block_tables, pre.prefix + pre.new)
    dk, dvv = dev(kk), dev(vv)
    bt, cu_q, cu_k = dev_i32(pre.block_tables), dev_i32(pre.cu_seqlens_q), dev_i32(
        pre.cu_seqlens_k)
    o = torch.empty(q.shape, dtype=torch.bfloat16, device=dev_t)
    sched = torch.zeros(1, dtype=torch.int32, device=dev_t)
    mq, mk = int(pre.new.max()), int((pre.prefix + pre.new).max())
    calls = {
        "paged": lambda: nv.nv_prefill_attn_paged(q, kc, vc, bt, o, cu_q, cu_k, mq, SCALE,
                                                  sched_counter=sched),
        "contiguous": lambda: nv.nv_prefill_attn_varlen(q, dk, dvv, o, cu_q, cu_k, mq, mk,
                                                        SCALE, sched_counter=sched),
    }
    out = {"workload": "qwen3_8b_16seq_prefix256x1-16_new128-1024", "tokens_new": int(L.sum()),
           "tokens_cached": int(P.sum()), "flops": flops}
    for name, fn in calls.items():
        times = []
        for i in range(reps + 3):
            flush()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            if i >= 3:
                times.append(e0.elapsed_time(e1) / 1e3)
        t = statistics.median(times)
        out[name] = {"ms": t * 1e3, "tflops": flops / t / 1e12,
                     "frac": flops / t / 1e12 / measured_peaks()[1]}
    del flush, kc, vc, dk, dvv
    return out


# ------------------------------------------ launch overhead: CUDA graph
def graph_decode_overhead(dev_t, buckets=(1, 8, 64, 512), ctx_len: int = 1024, reps: int = 100):
    """The decode layer's four ABI calls (Qwen3-8B heads) timed eagerly and as
    one captured CUDA graph per batch bucket, two ways: back to back (CUDA
    events over `reps` steps; eager steps then overlap through programmatic
    launch) and one step at a time with a read-back of the output (host clock;
    what a serving loop sees per step).  Every sequence has ctx_len keys;
    buckets above 2 end with two padded rows (slot -1, context length 0)."""
    import torch
    import paged_kv_attention_kvcache_gb300 as nv
    s = wl.QWEN3_8B
    nmax = max(buckets)
    blocks = -(-ctx_len // wl.BLOCK_SIZE)
    step = wl.make_decode(77, s, np.full(nmax, ctx_len, np.int32), nmax * blocks + 2,
                          with_norms=True, name="graph")
    Q, D = s.q_size, s.kv_size

    def dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(
            torch.bfloat16).to(dev_t)

    table = torch.empty(wl.MAX_POSITION, 128, dtype=torch.float32, device=dev_t)
    nv.nv_rope_cos_sin_cache(table, wl.ROPE_BASE)
    kc, vc = dev(step.pool.k), dev(step.pool.v)
    g, qn, kn = dev(step.gamma), dev(step.q_norm_w), dev(step.k_norm_w)
    out = []
    for b in buckets:
        n_real = b - 2 if b > 2 else b
        ctx = step.context_lens[:b].copy()
        slots = step.slot_mapping[:b].copy()
        ctx[n_real:] = 0
        slots[n_real:] = -1
        x, r = dev(step.x[:b]), dev(step.residual[:b])
        y = torch.empty_like(x)
        qkv = dev(step.qkv[:b])
        d_pos = torch.from_numpy(step.positions[:b].copy()).to(dev_t)
        d_slots = torch.from_numpy(slots).to(dev_t)
        d_bt = torch.from_numpy(step.block_tables[:b].copy()).to(dev_t)
        d_ctx = torch.from_numpy(ctx).to(dev_t)
        o = torch.empty(b, s.hq, 128, dtype=torch.bfloat16, device=dev_t)
        wsb = nv.nv_decode_attn_workspace_size(b, s.hq, s.hkv, 128, d_bt.shape[1],
                                               wl.BLOCK_SIZE, 0)
        ws = torch.empty(max(1, wsb // 4), dtype=torch.float32, device=dev_t)
        q = qkv[:, :Q].view(b, s.hq, 128)
        k = qkv[:, Q:Q + D].view(b, s.hkv, 128)
        v = qkv[:, Q + D:].view(b, s.hkv, 128)

        def layer():
            nv.nv_add_rmsnorm(x, r, g, y, r, eps=wl.RMS_EPS)
            nv.nv_qknorm_rope(q, k, qn, kn, table, d_pos, eps=wl.RMS_EPS)
            nv.nv_store_kvcache(k, v, kc, vc, d_slots)
            nv.nv_decode_attn_paged(q, kc, vc, d_bt, d_ctx, o, SCALE, workspace=ws)

        side = torch.cuda.Stream(device=dev_t)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(3):
                layer()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            layer()

        def timed(fn):
            for _ in range(10):
                fn()
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(reps):
                fn()
            e1.record()
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) * 1e3 / reps

        # One step at a time, as a serving loop runs it: launch the step, read
        # a few of its outputs back to the host and wait for them; host wall
        # clock, median.  Host launch cost and the step's full latency count
        # here; nothing overlaps across steps.
        host_o = torch.empty(8, dtype=torch.bfloat16).pin_memory()
        cur = torch.cuda.current_stream()

        def one_step(fn):
            fn()
            host_o.copy_(o.view(-1)[:8], non_blocking=True)
            cur.synchronize()

        def latency(fn, n=200):
            for _ in range(10):
                one_step(fn)
            ts = []
            for _ in range(n):
                t = time.perf_counter()
                one_step(fn)
                ts.append(time.perf_counter() - t)
            return statistics.median(ts) * 1e6

        eager_us = timed(layer)
        graph_us = timed(graph.replay)
        out.append({"bucket": b, "real": n_real, "eager_us": round(eager_us, 2),
                    "graph_us": round(graph_us, 2),
                    "eager_step_sync_us": round(latency(layer), 2),
                    "graph_step_sync_us": round(latency(graph.replay), 2),
                    "kernels": 4 + (1 if wsb else 0)})
        del graph
    return {"ctx": ctx_len, "heads": "32/8", "per_bucket": out}


# ------------------------------------------------------------ oracle side
def oracle_decode_step(step: wl.DecodeStep):
    """The fp64 oracle on the whole decode step: add-RMSNorm, QK-Norm + RoPE
    of q and k, store_kvcache of the new rows and paged decode of every
    (sequence, head).  Returns (seconds, threads)."""
    import oracle
    s = step.shape
    B = step.context_lens.size
    Q, D = s.q_size, s.kv_size
    t0 = time.time()
    oracle.add_rmsnorm(step.x, step.residual, step.gamma, wl.RMS_EPS)
    qb = step.qkv[:, :Q].reshape(B, s.hq, 128)
    kb = step.qkv[:, Q:Q + D].reshape(B, s.hkv, 128)
    vb = step.qkv[:, Q + D:].reshape(B, s.hkv, 128)
    q_rot = oracle.round_to_bf16(oracle.qknorm_rope(qb, step.q_norm_w, step.positions))
    k_rot = oracle.round_to_bf16(oracle.qknorm_rope(kb, step.k_norm_w, step.positions))
    oracle.store_kvcache(k_rot, vb, step.pool.k, step.pool.v, step.slot_mapping)
    oracle.paged_decode(q_rot, step.pool.k, step.pool.v, step.block_tables, step.context_lens,
                        SCALE)
    return time.time() - t0, oracle.num_threads()


def oracle_store_decode(step: wl.DecodeStep):
    """The oracle on a decode step without the norms: store_kvcache of the new
    token's K/V, then paged decode.  Returns seconds."""
    import oracle
    s = step.shape
    B = step.context_lens.size
    Q, D = s.q_size, s.kv_size
    t0 = time.time()
    oracle.store_kvcache(step.qkv[:, Q:Q + D].reshape(B, s.hkv, 128),
                         step.qkv[:, Q + D:].reshape(B, s.hkv, 128), step.pool.k, step.pool.v,
                         step.slot_mapping)
    oracle.paged_decode(step.qkv[:, :Q].reshape(B, s.hq, 128), step.pool.k, step.pool.v,
                        step.block_tables, step.context_lens, SCALE)
    return time.time() - t0


def repeat_for(fn, min_seconds: float):
    """Call fn() (which returns its own seconds) until min_seconds have been
    spent; returns (calls, seconds)."""
    n, total = 0, 0.0
    while n == 0 or total < min_seconds:
        total += fn()
        n += 1
    return n, total


def oracle_baseline(step: wl.DecodeStep, min_seconds: float = 10.0):
    """Repeat the oracle's decode step until at least min_seconds of work."""
    nbytes = decode_step_bytes(step)["total"]
    times, threads = [], 1
    while not times or sum(times) < min_seconds:
        dt, threads = oracle_decode_step(step)
        times.append(dt)
    return nbytes * len(times) / sum(times) / 1e9, threads, len(times), sum(times)


def visible_keys(cu_q: np.ndarray, cu_k: np.ndarray) -> np.ndarray:
    """Keys each packed query token sees under causality aligned to the last
    key: i + (Lk - Lq) + 1 for query i of its sequence."""
    lq = np.diff(cu_q).astype(np.int64)
    lk = np.diff(cu_k).astype(np.int64)
    seq = np.repeat(np.arange(lq.size), lq)
    i = np.arange(int(cu_q[-1]), dtype=np.int64) - cu_q[:-1].astype(np.int64)[seq]
    return i + (lk - lq)[seq] + 1


def oracle_attention_rate(call, vis: np.ndarray, hq: int, min_seconds: float, seed: int,
                          chunk: int = 4096):
    """TFLOP/s of the oracle's attention over credited row samples: chunks of
    `chunk` random (token, head) rows, each credited with its own causal
    pairs (4 * 128 * visible keys), until min_seconds of work.  `call(rows)`
    runs the oracle on the rows.  Returns (tflops, rows, seconds)."""
    g = np.random.default_rng(seed)
    flops, total, n = 0.0, 0.0, 0
    while n == 0 or total < min_seconds:
        toks = g.integers(0, vis.size, chunk)
        rows = np.stack([toks, g.integers(0, hq, chunk)], axis=1).astype(np.int64)
        t0 = time.time()
        call(rows)
        total += time.time() - t0
        flops += 4.0 * 128 * float(vis[toks].sum())
        n += chunk
    return flops / total / 1e12, n, total


def oracle_figures(r: dict, min_seconds: float = 4.0) -> dict:
    """The fp64 oracle timed on the host cores beside every throughput of the
    bench line other than the headline decode step, in the same units.  Each
    is a bounded sample, described in its `sample` field."""
    import oracle
    threads = oracle.num_threads()
    out = {}
    pre = r["pre"]
    s = pre.shape
    T, Q, D = pre.qkv.shape[0], s.q_size, s.kv_size
    q = pre.qkv[:, :Q].reshape(T, s.hq, 128)
    k = pre.qkv[:, Q:Q + D].reshape(T, s.hkv, 128)
    v = pre.qkv[:, Q + D:].reshape(T, s.hkv, 128)
    cu = pre.cu_seqlens
    # ---- prefill attention (cfg4 batch), credited rows
    tf, n, secs = oracle_attention_rate(
        lambda rows: oracle.attention_varlen(q, k, v, cu, cu, SCALE, True, rows=rows),
        visible_keys(cu, cu), s.hq, min_seconds, 7001)
    out["prefill_attention"] = {
        "value": tf, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
        "sample": f"{n} random (token, head) rows of the 33k-token batch, each credited with "
                  f"its causal pairs; {secs:.1f} s"}
    # ---- the prefill layer's other ops on the whole batch, then tokens/s of the
    # layer with attention at the rate just measured
    t0 = time.time()
    oracle.add_rmsnorm(pre.x, pre.residual, pre.gamma, wl.RMS_EPS)
    oracle.qknorm_rope(q, pre.q_norm_w, pre.positions)
    k_rot = oracle.round_to_bf16(oracle.qknorm_rope(k, pre.k_norm_w, pre.positions))
    kc = np.zeros((pre.num_blocks, wl.BLOCK_SIZE, s.hkv, 128), np.uint16)
    vc = np.zeros_like(kc)
    oracle.store_kvcache(k_rot, v, kc, vc, pre.slot_mapping)
    t_elem = time.time() - t0
    t_attn = prefill_flops(pre.lengths) / (tf * 1e12)
    out["prefill_layer_tokens_per_s"] = {
        "value": T / (t_elem + t_attn), "unit": "tokens/s", "cores": threads, "kind": "oracle",
        "sample": f"add-RMSNorm, QK-Norm+RoPE and store_kvcache of all {T} tokens timed "
                  f"({t_elem:.1f} s); attention at the sampled rate above"}
    # ---- QK-Norm + RoPE + store on the prefill batch (the fused pass's bytes)
    t0 = time.time()
    oracle.qknorm_rope(q, pre.q_norm_w, pre.positions)
    k_rot = oracle.round_to_bf16(oracle.qknorm_rope(k, pre.k_norm_w, pre.positions))
    oracle.store_kvcache(k_rot, v, kc, vc, pre.slot_mapping)
    t_rs = time.time() - t0
    out["rope_store_prefill"] = {
        "value": r["rope_store"]["fused_bytes"] / t_rs / 1e9, "unit": "GB/s", "cores": threads,
        "kind": "oracle", "sample": f"QK-Norm+RoPE of q and k, store_kvcache, all {T} tokens, "
                                    f"credited with the fused pass's bytes; {t_rs:.1f} s"}
    del kc, vc
    # ---- SiluAndMul, credited rows of the [T, 2 x 12288] activation
    inter = 12288
    xs = wl.normal_bf16(830, "bench.swiglu", (1024, 2 * inter))

    def swiglu():
        t0 = time.time()
        oracle.silu_and_mul(xs)
        return time.time() - t0

    calls, secs = repeat_for(swiglu, min_seconds / 2)
    out["silu_and_mul_prefill"] = {
        "value": calls * 1024 * 3 * inter * 2 / secs / 1e9, "unit": "GB/s", "cores": threads,
        "kind": "oracle", "sample": f"1024 rows x 12288 repeated {calls}x ({secs:.1f} s), "
                                    f"credited with 3 x 2 bytes per element"}
    # ---- decode sets
    st2 = wl.config2()
    nb2 = store_decode_bytes(st2)
    calls, secs = repeat_for(lambda: oracle_store_decode(st2), min_seconds)
    B2 = st2.context_lens.size
    out["b64_ctx512_4096_qwen3_06b_step"] = {
        "value": nb2["total"] * calls / secs / 1e9, "unit": "GB/s",
        "tokens_per_s": B2 * calls / secs, "cores": threads, "kind": "oracle",
        "sample": f"store_kvcache + paged decode of all 64 sequences, {calls}x ({secs:.1f} s)"}
    del st2
    st5 = wl.config5()
    nb5 = store_decode_bytes(st5)["attn"]
    B5 = st5.context_lens.size
    qb5 = st5.qkv[:, :st5.shape.q_size].reshape(B5, st5.shape.hq, 128)

    def dec5():
        t0 = time.time()
        oracle.paged_decode(qb5, st5.pool.k, st5.pool.v, st5.block_tables, st5.context_lens,
                            SCALE)
        return time.time() - t0

    calls, secs = repeat_for(dec5, min_seconds)
    out["b32_ctx4096_40960_qwen3_8b"] = {
        "value": nb5 * calls / secs / 1e9, "unit": "GB/s", "tokens_per_s": B5 * calls / secs,
        "cores": threads, "kind": "oracle",
        "sample": f"paged decode of all 32 sequences (unsplit), {calls}x ({secs:.1f} s)"}
    del st5
    # ---- prefill over the paged cache (prefix hit), credited rows
    px = wl.config_prefix()
    tf, n, secs = oracle_attention_rate(
        lambda rows: oracle.attention_paged_prefill(px.q, px.pool.k, px.pool.v, px.block_tables,
                                                    px.cu_seqlens_q, px.cu_seqlens_k, SCALE,
                                                    rows=rows),
        visible_keys(px.cu_seqlens_q, px.cu_seqlens_k), px.shape.hq, min_seconds, 7002)
    out["prefill_paged_prefix"] = {
        "value": tf, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
        "sample": f"{n} random (token, head) rows of the prefix-hit workload, each credited "
                  f"with its causal pairs; {secs:.1f} s"}
    return out


def slice_decode_step(step: wl.DecodeStep, idx: np.ndarray) -> wl.DecodeStep:
    """The same decode step restricted to the sequences `idx` (every op of the
    step is independent per sequence)."""
    import dataclasses

    def pick(a):
        return None if a is None else a[idx]
    return dataclasses.replace(step, context_lens=step.context_lens[idx],
                               positions=step.positions[idx], block_tables=step.block_tables[idx],
                               slot_mapping=step.slot_mapping[idx], qkv=step.qkv[idx],
                               x=pick(step.x), residual=pick(step.residual))


def run_reference(args, budget_s: float = 150.0):
    """The CPU reference arm: the fp64 oracle, as it stands, on the bench's
    workload.  Each step is the decode layer step (the line's value) and a
    sample of the prefill layer: one chunk of 2048 random (token, head)
    attention rows of the 33k-token batch, credited with their causal pairs.
    One untimed pass of the whole decode step sizes the run: if `steps` whole
    passes would take longer than `budget_s`, each step takes a rotating slice
    of the sequences (a bounded sample) credited with that slice's bytes."""
    import oracle
    oracle.build()
    step = wl.config3()
    pre = wl.config4()
    s = pre.shape
    T, Q, D = pre.qkv.shape[0], s.q_size, s.kv_size
    pq = pre.qkv[:, :Q].reshape(T, s.hq, 128)
    pk = pre.qkv[:, Q:Q + D].reshape(T, s.hkv, 128)
    pv = pre.qkv[:, Q + D:].reshape(T, s.hkv, 128)
    cu = pre.cu_seqlens
    vis = visible_keys(cu, cu)
    B = step.context_lens.size
    t_full, threads = oracle_decode_step(step)
    per = B
    if args.steps * t_full > budget_s:
        per = max(8, min(B, int(B * budget_s / (args.steps * t_full))))
    g = np.random.default_rng(7003)
    times, ptimes, nbytes, pflops = [], [], 0, 0.0
    for k in range(args.steps):
        sub = step if per == B else slice_decode_step(step, (k * per + np.arange(per)) % B)
        dt, threads = oracle_decode_step(sub)
        times.append(dt)
        nbytes += decode_step_bytes(sub)["total"]
        toks = g.integers(0, T, 2048)
        rows = np.stack([toks, g.integers(0, s.hq, 2048)], axis=1).astype(np.int64)
        t0 = time.time()
        oracle.attention_varlen(pq, pk, pv, cu, cu, SCALE, True, rows=rows)
        ptimes.append(time.time() - t0)
        pflops += 4.0 * 128 * float(vis[toks].sum())
    value = nbytes / sum(times) / 1e9
    ptf = pflops / sum(ptimes) / 1e12
    sample = (f"decode layer step (32 heads, ctx~U[1024,8192]): add-RMSNorm, QK-Norm+RoPE, "
              f"store_kvcache, paged decode; {per} of its {B} sequences per step"
              + (" (rotating slice), credited with their own bytes" if per < B else "")
              + "; plus 2048 random prefill attention rows per step, credited with their "
                "causal pairs")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * (sum(times) + sum(ptimes)) / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "global_batch": 256, "seq_len": SEQ_LEN,
                   "parallelism": "single", "decode_step_bytes": decode_step_bytes(step)["total"],
                   "timed": "the decode layer step (the line's value) and a sample of the "
                            "prefill layer's attention, in the fp64 CPU oracle"},
        "prefill": {"metric": "prefill attn TFLOP/s (causal pairs)", "value": ptf,
                    "unit": "TFLOP/s"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def run_ncu_case(which: str, launches: int = 3):
    """A small case of one kernel for detailed ncu captures: a few GB on the
    device at most, inputs above L2 size, `launches` calls of the op."""
    import torch
    import __graft_entry__
    import paged_kv_attention_kvcache_gb300 as nv
    __graft_entry__.build()
    torch.cuda.set_device(0)

    def dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(
            torch.bfloat16).cuda()

    if which == "decode-small":
        # The Qwen3-0.6B-head set as measured (B = 64, ctx U[512, 4096], 0.6 GB of
        # K/V, automatic split): store_kvcache of the new tokens, then decode.
        step = wl.config2()
        s = step.shape
        B, Q, D = step.context_lens.size, s.q_size, s.kv_size
        qkv = dev(step.qkv)
        q = qkv[:, :Q].view(B, s.hq, 128)
        k = qkv[:, Q:Q + D].view(B, s.hkv, 128)
        v = qkv[:, Q + D:].view(B, s.hkv, 128)
        kc, vc = dev(step.pool.k), dev(step.pool.v)
        bt = torch.from_numpy(step.block_tables).cuda()
        cl = torch.from_numpy(step.context_lens).cuda()
        slots = torch.from_numpy(step.slot_mapping).cuda()
        o = torch.empty(B, s.hq, 128, dtype=torch.bfloat16, device="cuda")
        ws_b = nv.nv_decode_attn_workspace_size(B, s.hq, s.hkv, 128, bt.shape[1], 256, 0)
        ws = torch.empty(max(1, ws_b // 4), dtype=torch.float32, device="cuda")
        for _ in range(launches):
            nv.nv_store_kvcache(k, v, kc, vc, slots)
            nv.nv_decode_attn_paged(q, kc, vc, bt, cl, o, SCALE, workspace=ws)
    elif which == "decode":
        # Qwen3-8B heads, 64 sequences of 8192 keys: 2.1 GB of K/V, split as the
        # bench's decode step is (2048 keys).
        ctx = np.full(64, 8192, np.int32)
        step = wl.make_decode(9, wl.QWEN3_8B, ctx, 64 * 32 + 8, with_norms=False,
                              name="ncu.decode")
        s = step.shape
        q = dev(step.qkv[:, :s.q_size]).view(64, s.hq, 128)
        kc, vc = dev(step.pool.k), dev(step.pool.v)
        bt = torch.from_numpy(step.block_tables).cuda()
        cl = torch.from_numpy(step.context_lens).cuda()
        o = torch.empty(64, s.hq, 128, dtype=torch.bfloat16, device="cuda")
        ws_b = nv.nv_decode_attn_workspace_size(64, s.hq, s.hkv, 128, bt.shape[1], 256, 0)
        ws = torch.empty(max(1, ws_b // 4), dtype=torch.float32, device="cuda")
        for _ in range(launches):
            nv.nv_decode_attn_paged(q, kc, vc, bt, cl, o, SCALE, workspace=ws)
    else:
        # Qwen3-8B heads, 8 sequences of 2048 tokens (0.2 GB of q/k/v).
        lengths = np.full(8, 2048, np.int64)
        pre = wl.make_prefill(9, wl.QWEN3_8B, lengths, name="ncu.prefill")
        s = pre.shape
        T = int(lengths.sum())
        qkv = dev(pre.qkv)
        Q, D = s.q_size, s.kv_size
        q, k, v = (qkv[:, :Q].view(T, s.hq, 128), qkv[:, Q:Q + D].view(T, s.hkv, 128),
                   qkv[:, Q + D:].view(T, s.hkv, 128))
        cu = torch.from_numpy(pre.cu_seqlens).cuda()
        o = torch.empty(T, s.hq, 128, dtype=torch.bfloat16, device="cuda")
        sched = torch.zeros(1, dtype=torch.int32, device="cuda")
        for _ in range(launches):
            nv.nv_prefill_attn_varlen(q, k, v, o, cu, cu, 2048, 2048, SCALE, sched_counter=sched)
    torch.cuda.synchronize()
    print(f"ncu case {which}: {launches} launches done")


def run_ncu_layer_case(launches: int = 2):
    """Every kernel of the Qwen3-8B prefill layer on the bench batch (33,109
    tokens), plus the fused rope+store pass and SiluAndMul (I = 12288), each
    `launches` times: ~3 GB on the device, inputs above L2 size."""
    import torch
    import __graft_entry__
    import paged_kv_attention_kvcache_gb300 as nv
    __graft_entry__.build()
    torch.cuda.set_device(0)

    def dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(
            torch.bfloat16).cuda()

    pre = wl.config4()
    s = pre.shape
    T, Q, D = pre.qkv.shape[0], s.q_size, s.kv_size
    table = torch.empty(wl.MAX_POSITION, 128, dtype=torch.float32, device="cuda")
    nv.nv_rope_cos_sin_cache(table, wl.ROPE_BASE)
    x, r, g = dev(pre.x), dev(pre.residual), dev(pre.gamma)
    y = torch.empty_like(x)
    qkv = dev(pre.qkv)
    q, k, v = (qkv[:, :Q].view(T, s.hq, 128), qkv[:, Q:Q + D].view(T, s.hkv, 128),
               qkv[:, Q + D:].view(T, s.hkv, 128))
    qn, kn = dev(pre.q_norm_w), dev(pre.k_norm_w)
    pos = torch.from_numpy(pre.positions).cuda()
    slots = torch.from_numpy(pre.slot_mapping).cuda()
    cu = torch.from_numpy(pre.cu_seqlens).cuda()
    kc = torch.zeros(pre.num_blocks, wl.BLOCK_SIZE, s.hkv, 128, dtype=torch.bfloat16,
                     device="cuda")
    vc = torch.zeros_like(kc)
    o = torch.empty(T, s.hq, 128, dtype=torch.bfloat16, device="cuda")
    sched = torch.zeros(1, dtype=torch.int32, device="cuda")
    ml = int(pre.lengths.max())
    gate_up = torch.empty(T, 2 * 12288, dtype=torch.bfloat16, device="cuda").normal_()
    act = torch.empty(T, 12288, dtype=torch.bfloat16, device="cuda")
    for _ in range(launches):
        nv.nv_add_rmsnorm(x, r, g, y, r, eps=wl.RMS_EPS)
        nv.nv_qknorm_rope(q, k, qn, kn, table, pos, eps=wl.RMS_EPS)
        nv.nv_store_kvcache(k, v, kc, vc, slots)
        nv.nv_prefill_attn_varlen(q, k, v, o, cu, cu, ml, ml, SCALE, sched_counter=sched)
        nv.nv_qknorm_rope_store(q, k, v, qn, kn, table, pos, kc, vc, slots, eps=wl.RMS_EPS,
                                write_k=True)
        nv.nv_silu_and_mul(gate_up, act)
    torch.cuda.synchronize()
    print(f"ncu case layer: {launches} launches of each kernel done")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ncu-case", choices=["decode", "decode-small", "prefill", "layer"],
                    default=None,
                    help="run a small case of one kernel, or every prefill-layer kernel on the "
                         "bench batch (for ncu captures), and exit")
    args = ap.parse_args()
    if args.ncu_case == "layer":
        run_ncu_layer_case()
        return
    if args.ncu_case:
        run_ncu_case(args.ncu_case)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            run_reference(args)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    import __graft_entry__
    __graft_entry__.build()
    r = run_ours(args, rank, world, local_rank)

    # The oracle is timed on the host cores beside a single-GPU run only; with
    # several replicas the line reports the GPUs alone.
    cpu = None
    ofig = {}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        val, threads, reps, secs = oracle_baseline(r["step"])
        cpu = {"value": val, "unit": "GB/s", "cores": threads, "kind": "oracle",
               "tokens_per_s": r["step"].context_lens.size * reps / secs,
               "sample": f"whole decode step (256 seqs x 32 heads: add-RMSNorm, QK-Norm+RoPE, "
                         f"store_kvcache, paged decode) repeated {reps}x, {secs:.1f} s of CPU "
                         f"time"}
        ofig = oracle_figures(r)
        r["decode_sets"]["b64_ctx512_4096_qwen3_06b_step"]["oracle"] = \
            ofig["b64_ctx512_4096_qwen3_06b_step"]
        for key in ("b32_ctx4096_40960_qwen3_8b_splitauto", "b32_ctx4096_40960_qwen3_8b_split1024"):
            r["decode_sets"][key]["oracle"] = ofig["b32_ctx4096_40960_qwen3_8b"]
        r["prefix_prefill"]["oracle"] = ofig["prefill_paged_prefix"]
        r["rope_store"]["oracle"] = ofig["rope_store_prefill"]
        r["swiglu"]["oracle"] = ofig["silu_and_mul_prefill"]
    if rank == 0:
        nbytes = r["nbytes"]
        B_dec = r["step"].context_lens.size
        traffic = None
        if kernel_source_hash("decode_attn.cu") == DECODE_TRAFFIC["source_sha256_16"]:
            traffic = DECODE_TRAFFIC["ratio"] * nbytes["attn"]
        line = {
            "metric": METRIC, "value": r["value"], "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {
                "workload": WORKLOAD,
                "global_batch": 256 * world, "seq_len": SEQ_LEN,
                "parallelism": "replicas" if world > 1 else "single",
                "decode_kv_bytes": nbytes["attn"], "decode_step_bytes": nbytes["total"],
                "prefill_tokens": r["T"], "l2": "flushed between steps (256 MB written, then another 256 MB read)",
                "decode_ms": r["dec_ms"], "prefill_ms": r["pre_ms"]},
            "roofline": {"bound": "hbm", "kernel": "nv_decode_attn_paged (split + merge)",
                         "achieved": r["attn_gbs"], "peak": r["hbm"], "unit": "GB/s",
                         "frac": r["attn_gbs"] / r["hbm"], "traffic": traffic,
                         "peak_source": r["peak_src"], "launch_ms": r["attn_ms"]},
            "prefill": {"metric": "prefill attn TFLOP/s (causal pairs)", "value": r["ptflops"],
                        "unit": "TFLOP/s", "launch_ms": r["pattn_ms"],
                        "oracle": ofig.get("prefill_attention"),
                        "roofline": {"bound": "tensor", "achieved": r["ptflops"],
                                     "peak": r["bf16"], "unit": "TFLOP/s",
                                     "frac": r["ptflops"] / r["bf16"],
                                     "traffic": (PREFILL_TRAFFIC["bytes"]
                                                 if kernel_source_hash("prefill_attn.cu")
                                                 == PREFILL_TRAFFIC["source_sha256_16"] else None),
                                     "traffic_unit": "bytes per launch",
                                     "peak_source": r["peak_src"] + " bf16 burst"}},
            "cpu_baseline": cpu,
            "e2e": {"value": r["e2e"], "unit": "GB/s", "h2d_bytes_per_step": r["h2d"],
                    "d2h_bytes_per_step": r["d2h"]},
            "tokens_per_s": {"decode": world * B_dec / (r["dec_ms"] / 1e3),
                             "prefill": world * r["T"] / (r["pre_ms"] / 1e3),
                             "oracle_decode": cpu["tokens_per_s"] if cpu else None,
                             "oracle_prefill": (ofig["prefill_layer_tokens_per_s"]["value"]
                                                if ofig else None),
                             "oracle_cores": cpu["cores"] if cpu else None},
            "nominal_frac": {"decode_attn_of_7900_GBs": r["attn_gbs"] / 7900.0,
                             "prefill_of_2250_TFLOPs": r["ptflops"] / 2250.0},
            "decode_attention_sets": r["decode_sets"],
            "prefill_paged_prefix": r["prefix_prefill"],
            "decode_graph": r["graph"],
            "rope_store_prefill": r["rope_store"],
            "silu_and_mul_prefill": r["swiglu"],
            "gpu_launches": r["launches"],
            "clocks": r["clocks"],
            "clock_block": r["clock_block"],
        }
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
