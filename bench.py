#!/usr/bin/env python
"""Decode-step benchmark of VQ KV-cache decode attention on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload I]

One step = the whole decode hot path for one batch, one vq_decode_step call:
encode the appended token of every sequence into the cache (slots from the
page table), split attention over the quantized cache and the split combine.
The default workload is Llama-3.1-8B layer shape, batch 1, 32 query / 8 KV
heads, 32768 cached tokens (+1 appended), 2-bit K and V codes (d = 4, 256
centroids).

Timing: W eager warm-up steps; then exactly K steps captured in one CUDA graph
and replayed between CUDA events, with a barrier and a synchronize on both
sides (max over ranks).  Step i reads cache copy i % R, R copies together
larger than twice the L2 cache, so codes come from HBM.  The roofline uses the
split kernel's average launch duration from a graph of K back-to-back split
launches (same rotation) between two events; a graph of the steps with event
nodes around every kernel gives the per-kernel breakdown (event nodes add their
own latency, so those figures run high).  SM clocks are sampled with
nvidia-smi during the load.

--impl reference times the fp64 CPU oracle (the correctness reference) on the
host cores on a bounded sample of the same workload; it is a deliberately slow
baseline, not a target.  Under torchrun only rank 0 runs it.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import re
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "decode-attn KV tokens/s and achieved HBM GB/s (% of 8 TB/s) on compressed KV"
UNIT = "KV tokens/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
CALIB_DIR = os.path.join(ROOT, "tests", "golden", "calib")
KERNEL_SRCS = [os.path.join(ROOT, "bit_vector_quantized_gb300", "csrc", f)
               for f in ("vq_decode_kernel.cuh", "vq_decode.cu", "vq_decode_balanced.cu",
                         "vq_device.cuh", "vq_kernels.h")]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_split_traffic.json")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=1)
    ap.add_argument("--copies", type=int, default=0, help="rotating cache copies (0: auto)")
    ap.add_argument("--splits", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--soak-seconds", type=float, default=1.5)
    ap.add_argument("--no-fp16-compare", action="store_true",
                    help="skip the dense fp16 attention comparison (context only)")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="skip the long-context and large-batch split-kernel blocks")
    ap.add_argument("--no-methods", action="store_true",
                    help="skip the score / P.V method comparison (gather, LUT, bins)")
    ap.add_argument("--methods-only", action="store_true",
                    help="launch the split kernel three times per method on the workload and "
                         "exit (a short program for an ncu capture of the three methods)")
    ap.add_argument("--launches-only", action="store_true",
                    help="launch the split kernel alone four times, then the decode step four "
                         "times, on the workload (seeded random codes) and exit (a short program "
                         "for ncu captures of either)")
    return ap.parse_args()


def load_calib(i):
    z = np.load(os.path.join(CALIB_DIR, f"cfg{i}.npz"))
    return z["lam"], z["ck"], z["cv"]


def step_launches(w, sms):
    """Kernels one vq_decode_step launches (include/vqattn.h).  With at most
    one sequence-KV-head pair per SM the attention kernel appends the new
    tokens itself: two kernels (with the merge), or three for the 1.5-bit
    format (its sliced codebook scan first).  Otherwise the append encode, the
    attention kernel and the merge, with one more (the candidates' merge) for
    10- to 12-bit codebooks."""
    wide = max(w.k_bits, w.v_bits) >= 10
    if w.batch * w.num_kv_heads <= sms:
        if w.k_bits <= 9 and w.v_bits <= 9:
            return 2
        if w.k_sub == 8 and w.k_bits == 12 and w.v_sub == 8 and w.v_bits == 12:
            return 3
    return 4 if wide else 3


def tokens_per_step(w):
    return int((W.seq_lens(w) + 1).sum())


def code_bytes_per_step(w):
    return tokens_per_step(w) * w.num_kv_heads * (w.k_code_bytes() + w.v_code_bytes())


def measured_hbm():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_hash():
    """sha256[:16] of the split kernel's code: its source file and the headers it
    includes, without comments and blank lines (an edited comment keeps a traffic
    record; any code change drops it)."""
    lines = []
    for path in KERNEL_SRCS:
        with open(path) as f:
            text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        lines += [ln.rstrip() for ln in text.splitlines() if ln.strip()]
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()[:16]


def recorded_traffic(workload):
    """DRAM bytes per split launch from a committed ncu summary, if current."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
        if t.get("kernel_sha256_16") == kernel_hash() and int(t.get("workload", -1)) == workload:
            return float(t["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


# ----------------------------------------------------------------- clocks ---

class ClockSampler:
    QUERY = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_id: str):
        self.path = tempfile.mktemp(prefix="vq_clocks_", suffix=".csv")
        self.proc = None
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", device_id, f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def device_id_for_smi(torch, dev):
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        return vis.split(",")[dev] if vis else str(dev)


# -------------------------------------------------------------- CPU oracle ---

def oracle_step_sampler(w, lam, ck, cv, n_sample):
    """Returns (step_fn, tokens attended per step) for an oracle decode step on a sample.

    Sample: sequence 0, all KV heads, the first n_sample cached tokens plus the
    appended token.  The step encodes the appended token (all KV heads) and runs
    decode attention for every query head over n_sample + 1 tokens.
    """
    import oracle
    n_sample = int(min(n_sample, W.seq_lens(w)[0]))
    k = W.kv_tokens(w, 0, "k", 0, n_sample)
    v = W.kv_tokens(w, 0, "v", 0, n_sample)
    lam64 = lam.astype(np.float64)
    kc, _, _, _ = oracle.encode_keys(k, lam64, ck, w.k_sub)       # the cached prefix
    vc, _, _, _ = oracle.encode_values(v, cv, w.v_sub)
    n = int(W.seq_lens(w)[0])
    k_new = W.kv_tokens(w, 0, "k", n, n + 1)
    v_new = W.kv_tokens(w, 0, "v", n, n + 1)
    q = W.queries(w)[0]

    def step():
        kn, _, _, _ = oracle.encode_keys(k_new, lam64, ck, w.k_sub)
        vn, _, _, _ = oracle.encode_values(v_new, cv, w.v_sub)
        return oracle.decode_attention(q, lam64, np.concatenate([kc, kn]), ck,
                                       np.concatenate([vc, vn]), cv)
    return step, n_sample + 1


def run_cpu_baseline(w, lam, ck, cv, seconds):
    import oracle
    oracle.set_num_threads(os.cpu_count() or 1)
    n_sample = min(2048, int(W.seq_lens(w)[0]))
    step, toks = oracle_step_sampler(w, lam, ck, cv, n_sample)
    step()
    t0 = time.perf_counter()
    n = 0
    while True:
        step()
        n += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = (time.perf_counter() - t0) / n
    cores = oracle.num_threads()
    # the same sample on one thread, for a quarter of the time
    oracle.set_num_threads(1)
    step()
    t1 = time.perf_counter()
    n1 = 0
    while True:
        step()
        n1 += 1
        if time.perf_counter() - t1 >= seconds / 4:
            break
    dt1 = (time.perf_counter() - t1) / n1
    oracle.set_num_threads(cores)
    return {"value": toks / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"sequence 0, all {w.num_kv_heads} KV heads / {w.num_q_heads} query heads, "
                      f"first {toks - 1} cached tokens + 1 appended (append encode + attention); "
                      f"{n} steps in {n * dt:.1f} s; per-token rate equals the full-context rate",
            "ms_per_sample_step": dt * 1e3,
            "single_thread": {"value": toks / dt1, "unit": UNIT, "cores": 1,
                              "ms_per_sample_step": dt1 * 1e3}}


def run_reference(args, w, rank):
    if rank != 0:
        return
    import oracle
    lam, ck, cv = load_calib(args.workload)
    oracle.set_num_threads(os.cpu_count() or 1)
    budget = 150.0
    probe_n = min(256, int(W.seq_lens(w)[0]))
    step, toks = oracle_step_sampler(w, lam, ck, cv, probe_n)
    step()
    t0 = time.perf_counter()
    step()
    per_tok = (time.perf_counter() - t0) / toks
    target = max(budget / max(args.steps + args.warmup, 1), 0.02)
    n_sample = int(max(64, min(int(W.seq_lens(w)[0]), target / max(per_tok, 1e-9))))
    step, toks = oracle_step_sampler(w, lam, ck, cv, n_sample)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / max(args.steps, 1)
    value = toks / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, None, None),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                         "kind": "oracle",
                         "sample": f"sequence 0, all KV heads, first {toks - 1} cached tokens + 1 "
                                   f"appended per step (append encode + attention)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def fp16_comparison(torch, w, dev, steps, l2):
    """Context, not the product path: PyTorch's scaled_dot_product_attention
    (a library kernel) for one decode query per sequence over dense fp16 K/V of
    the same shape (every sequence padded to the longest; GQA), timed like the
    step: a CUDA graph of `steps` launches over rotating copies larger than L2."""
    import torch.nn.functional as F
    B, Hq, Hkv, D = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim
    N = int(W.seq_lens(w).max()) + 1
    kv_bytes = 2 * B * Hkv * N * D * 2
    copies = max(1, -(-2 * l2 // kv_bytes))
    if kv_bytes * copies > 24e9:
        return {"skipped": "dense fp16 K/V would not fit the memory budget"}
    g = torch.Generator(device=dev).manual_seed(0)
    q = torch.randn((B, Hq, 1, D), generator=g, device=dev, dtype=torch.float16)
    kvs = [(torch.randn((B, Hkv, N, D), generator=g, device=dev, dtype=torch.float16),
            torch.randn((B, Hkv, N, D), generator=g, device=dev, dtype=torch.float16)) for _ in range(copies)]

    def one(i):
        k, v = kvs[i % copies]
        return F.scaled_dot_product_attention(q, k, v, enable_gqa=True)

    for i in range(3):
        one(i)
    torch.cuda.synchronize()
    gr = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(gr, stream=s):
            for i in range(steps):
                one(i)
    torch.cuda.current_stream().wait_stream(s)
    gr.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    gr.replay()
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    del kvs
    torch.cuda.empty_cache()
    return {"kernel": "torch scaled_dot_product_attention, fp16 K/V, enable_gqa", "us_per_step": ms * 1e3,
            "kv_bytes_per_step": kv_bytes, "hbm_gbs": kv_bytes / (ms / 1e3) / 1e9,
            "padded_tokens_per_sequence": N}


def graph_ms(torch, dev, fn, steps):
    """Milliseconds per call of fn(i): 3 eager calls, then `steps` calls captured
    in one CUDA graph, replayed once to warm up and once between events."""
    for i in range(3):
        fn(i)
    torch.cuda.synchronize()
    gr = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(gr, stream=s):
            for i in range(steps):
                fn(i)
    torch.cuda.current_stream().wait_stream(s)
    gr.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    gr.replay()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def residual_comparison(torch, vq, w, layout, pools, lam_d, ck_d, cv_d, q_d, table_d, seq_d,
                        max_len, num_pages, splits, steps, dev, window=128):
    """Context: decode attention with the pages' full-precision residual window
    (实验结果 / 实验设置: 128 tokens) through vq_decode_attention_residual, against
    vq_decode_attention on the same quantized cache, timed like the step."""
    B, Hq, Hkv, D = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim
    g = torch.Generator(device=dev).manual_seed(0)
    k_res = torch.randn((B, Hkv, window, D), generator=g, device=dev, dtype=torch.float16)
    v_res = torch.randn((B, Hkv, window, D), generator=g, device=dev, dtype=torch.float16)
    res_lens = torch.full((B,), window, dtype=torch.int32, device=dev)
    ws_bytes = vq.vq_decode_residual_workspace_bytes(layout, B, max_len, splits)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    out = torch.empty((B, Hq, D), dtype=torch.float16, device=dev)
    copies = len(pools)
    p = lambda t: t.data_ptr()  # noqa: E731

    def plain(i):
        kp, vp = pools[i % copies]
        vq.vq_decode_attention(layout, B, p(q_d), p(lam_d), p(ck_d), p(cv_d), p(kp), p(vp), num_pages,
                               p(table_d), table_d.shape[1], p(seq_d), max_len, 0.0, splits, p(out),
                               p(ws), ws_bytes, None, torch.cuda.current_stream().cuda_stream)

    def with_window(i):
        kp, vp = pools[i % copies]
        vq.vq_decode_attention_residual(layout, B, p(q_d), p(lam_d), p(ck_d), p(cv_d), p(kp), p(vp),
                                        num_pages, p(table_d), table_d.shape[1], p(seq_d), max_len,
                                        p(k_res), p(v_res), p(res_lens), window, 0.0, splits, p(out),
                                        p(ws), ws_bytes, None, torch.cuda.current_stream().cuda_stream)

    plain_ms = graph_ms(torch, dev, plain, steps)
    window_ms = graph_ms(torch, dev, with_window, steps)
    return {"window_tokens": window, "attention_us": plain_ms * 1e3,
            "attention_with_window_us": window_ms * 1e3,
            "window_overhead_us": (window_ms - plain_ms) * 1e3}


def unfused_comparison(torch, vq, w, layout, pools, lam_d, ck_d, cv_d, q_d, num_pages, lens,
                       steps, dev):
    """Context, not the product path: the unfused pipeline VecInfer compares its
    fused kernel against (实验结果, 图5).  Every step dequantises the whole cache
    of every sequence to dense fp16 K^, V^ with vq_dequantize_kv (sequences
    padded to the longest, padding rows zero), then runs PyTorch's
    scaled_dot_product_attention (a library kernel, GQA) over them.  Timed like
    the step: a CUDA graph of `steps` launches over the rotating pool copies."""
    import torch.nn.functional as F
    B, Hq, Hkv, D = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim
    N = int(lens.max()) + 1
    dense_bytes = 2 * B * N * Hkv * D * 2
    if dense_bytes > 24e9:
        return {"skipped": "dense fp16 K/V would not fit the memory budget"}
    slots = np.full((B, N), -1, np.int64)
    for b, n in enumerate(lens):
        slots[b, :int(n) + 1] = W.slot_mapping(w, b, 0, int(n) + 1)
    slots_d = torch.from_numpy(slots.reshape(-1)).to(dev)
    k_hat = torch.empty((B * N, Hkv, D), dtype=torch.float16, device=dev)
    v_hat = torch.empty_like(k_hat)
    k4 = k_hat.view(B, N, Hkv, D).transpose(1, 2)
    v4 = v_hat.view(B, N, Hkv, D).transpose(1, 2)
    q4 = q_d.view(B, Hq, 1, D)
    copies = len(pools)

    def dequant(i):
        kp, vp = pools[i % copies]
        vq.vq_dequantize_kv(layout, B * N, slots_d.data_ptr(), lam_d.data_ptr(), ck_d.data_ptr(),
                            cv_d.data_ptr(), kp.data_ptr(), vp.data_ptr(), num_pages,
                            k_hat.data_ptr(), v_hat.data_ptr(), None,
                            torch.cuda.current_stream().cuda_stream)

    def one(i):
        dequant(i)
        return F.scaled_dot_product_attention(q4, k4, v4, enable_gqa=True)

    ms = graph_ms(torch, dev, one, steps)
    dq_ms = graph_ms(torch, dev, dequant, steps)
    code_bytes = B * N * Hkv * (layout_row_bytes(w, "k") + layout_row_bytes(w, "v"))
    del k_hat, v_hat, k4, v4
    torch.cuda.empty_cache()
    return {"pipeline": "vq_dequantize_kv, then torch scaled_dot_product_attention (fp16, enable_gqa)",
            "us_per_step": ms * 1e3, "dequantize_us": dq_ms * 1e3,
            "dequantize_gbs": (code_bytes + dense_bytes) / (dq_ms / 1e3) / 1e9,
            "dense_bytes_per_step": dense_bytes, "padded_tokens_per_sequence": N}


def layout_row_bytes(w, which):
    d, b = (w.k_sub, w.k_bits) if which == "k" else (w.v_sub, w.v_bits)
    return (-(-(w.head_dim // d) * b // 8) + 3) // 4 * 4


def split_kernel_block(torch, vq, wi, dev, steps, l2, hbm_peak, only_launch=False):
    """The decode step and the split attention kernel alone on another
    workload, timed like the headline: CUDA graphs of `steps` back-to-back
    calls rotating over cache copies larger than twice L2.  The pools hold
    seeded uniform random code bytes instead of an encoded prefill (which at
    these sizes would take minutes of host-side input generation): the
    kernel's work and memory traffic do not depend on the code values."""
    w = W.WORKLOADS[wi]
    lam, ck, cv = load_calib(wi)
    layout = vq.make_layout(w.head_dim, w.num_q_heads, w.num_kv_heads, w.k_sub, w.k_bits,
                            w.v_sub, w.v_bits, w.page_size)
    lens = (W.seq_lens(w) + 1).astype(np.int32)
    B, num_pages = w.batch, W.num_pages(w)
    table_d = torch.from_numpy(W.page_table(w)).to(dev)
    seq_d = torch.from_numpy(lens).to(dev)
    max_len = int(lens.max())
    step_bytes = code_bytes_per_step(w)
    copies = 1 if only_launch else max(1, -(-2 * l2 // step_bytes))
    gen = torch.Generator(device=dev).manual_seed(1000 + wi)
    krow, vrow = layout_row_bytes(w, "k"), layout_row_bytes(w, "v")
    pools = [(torch.randint(0, 256, (num_pages, w.num_kv_heads, w.page_size, krow), generator=gen,
                            device=dev, dtype=torch.uint8),
              torch.randint(0, 256, (num_pages, w.num_kv_heads, w.page_size, vrow), generator=gen,
                            device=dev, dtype=torch.uint8)) for _ in range(copies)]
    q_d = torch.from_numpy(W.queries(w)).to(dev)
    kv_new = torch.randn((2, B, w.num_kv_heads, w.head_dim), generator=gen, device=dev).half()
    lam_d, ck_d, cv_d = (torch.from_numpy(x).to(dev) for x in (lam, ck, cv))
    splits = vq.vq_default_num_splits(layout, B, max_len)
    ws_bytes = vq.vq_decode_workspace_bytes(layout, B, max_len, splits)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    out = torch.empty((B, w.num_q_heads, w.head_dim), dtype=torch.float16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    p = lambda t: t.data_ptr()  # noqa: E731

    def split_only(i):
        kp, vp = pools[i % copies]
        vq.vq_decode_partial(layout, B, p(q_d), p(lam_d), p(ck_d), p(cv_d), p(kp), p(vp), num_pages,
                             p(table_d), table_d.shape[1], p(seq_d), max_len, 0.0, splits, p(ws),
                             ws_bytes, p(status), torch.cuda.current_stream().cuda_stream)

    def step(i):
        kp, vp = pools[i % copies]
        vq.vq_decode_step(layout, B, p(q_d), p(kv_new[0]), p(kv_new[1]), p(lam_d), p(ck_d), p(cv_d),
                          p(kp), p(vp), num_pages, p(table_d), table_d.shape[1], p(seq_d), max_len,
                          0.0, splits, p(out), p(ws), ws_bytes, p(status),
                          torch.cuda.current_stream().cuda_stream)

    if only_launch:
        for fn in (split_only, step):
            for i in range(4):
                fn(i)
        torch.cuda.synchronize()
        return {"workload": w.name, "num_splits": splits, "device_status": int(status.item())}
    split_ms = graph_ms(torch, dev, split_only, steps)
    step_ms = graph_ms(torch, dev, step, steps)
    torch.cuda.synchronize()
    st = int(status.item())
    achieved = step_bytes / (split_ms / 1e3) / 1e9
    toks = int(lens.sum())
    res = {"workload": w.name, "num_splits": splits,
           "algorithmic_bytes_per_launch": step_bytes,
           "split_kernel_us": split_ms * 1e3, "achieved_gbs": achieved, "frac": achieved / hbm_peak,
           "pct_of_8tbs": 100 * achieved / NOMINAL_HBM_GBS,
           "step_us": step_ms * 1e3, "kv_tokens_per_s": toks / (step_ms / 1e3),
           "l2": f"rotating {copies} cache copies ({copies * step_bytes / 1e6:.0f} MB of codes)",
           "codes": "seeded uniform random bytes", "device_status": st}
    del pools, ws
    torch.cuda.empty_cache()
    return res


METHODS = {0: "gather", 1: "lut", 2: "bins"}


def method_comparison(torch, vq, wi, dev, steps, l2, hbm_peak, only_launch=False):
    """The split kernel with each of the pages' score / P.V methods
    (vq_decode_partial_method): in-register centroid gathers on the tensor
    cores (the library's), a per-query q~ x K-codebook lookup table for the
    scores (VecInfer, 内核实现细节 - 融合内核), and P.V through per-code bins
    (CommVQ, 降低计算复杂度).  Timed like the headline split kernel, over seeded
    random code bytes (the work and traffic do not depend on code values)."""
    w = W.WORKLOADS[wi]
    if not (w.k_sub == 4 and w.k_bits == 8 and w.v_sub == 4 and w.v_bits == 8
            and w.num_q_heads // w.num_kv_heads <= 4):
        return {"skipped": "the table-based methods are built for d = 4, 8-bit codes, G <= 4"}
    lam, ck, cv = load_calib(wi)
    layout = vq.make_layout(w.head_dim, w.num_q_heads, w.num_kv_heads, w.k_sub, w.k_bits,
                            w.v_sub, w.v_bits, w.page_size)
    lens = (W.seq_lens(w) + 1).astype(np.int32)
    B, num_pages = w.batch, W.num_pages(w)
    step_bytes = code_bytes_per_step(w)
    copies = 1 if only_launch else max(1, -(-2 * l2 // step_bytes))
    gen = torch.Generator(device=dev).manual_seed(2000 + wi)
    krow, vrow = layout_row_bytes(w, "k"), layout_row_bytes(w, "v")
    pools = [(torch.randint(0, 256, (num_pages, w.num_kv_heads, w.page_size, krow), generator=gen,
                            device=dev, dtype=torch.uint8),
              torch.randint(0, 256, (num_pages, w.num_kv_heads, w.page_size, vrow), generator=gen,
                            device=dev, dtype=torch.uint8)) for _ in range(copies)]
    table_d = torch.from_numpy(W.page_table(w)).to(dev)
    seq_d = torch.from_numpy(lens).to(dev)
    max_len = int(lens.max())
    q_d = torch.from_numpy(W.queries(w)).to(dev)
    lam_d, ck_d, cv_d = (torch.from_numpy(x).to(dev) for x in (lam, ck, cv))
    splits = vq.vq_default_num_splits(layout, B, max_len)
    ws_bytes = vq.vq_decode_workspace_bytes(layout, B, max_len, splits)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    p = lambda t: t.data_ptr()  # noqa: E731
    res = {"workload": w.name, "num_splits": splits, "codes": "seeded uniform random bytes"}
    for method, name in METHODS.items():
        def fn(i, method=method):
            kp, vp = pools[i % copies]
            vq.vq_decode_partial_method(layout, B, p(q_d), p(lam_d), p(ck_d), p(cv_d), p(kp), p(vp),
                                        num_pages, p(table_d), table_d.shape[1], p(seq_d), max_len,
                                        0.0, splits, method, p(ws), ws_bytes, p(status),
                                        torch.cuda.current_stream().cuda_stream)
        if only_launch:
            for i in range(3):
                fn(i)
            torch.cuda.synchronize()
            continue
        ms = graph_ms(torch, dev, fn, steps)
        gbs = step_bytes / (ms / 1e3) / 1e9
        res[name] = {"split_kernel_us": ms * 1e3, "achieved_gbs": gbs, "frac": gbs / hbm_peak}
    torch.cuda.synchronize()
    res["device_status"] = int(status.item())
    del pools, ws
    torch.cuda.empty_cache()
    return res


def encode_report(w, tokens, ms, sms, clocks):
    """Prefill encode throughput and its roofline.  The encode is bound by the FP32
    pipe: a nearest-centroid scan spends d fused multiply-adds per centroid and
    sub-vector, i.e. 2^bits * head_dim per token-head and tensor; the peak is
    128 FP32 lanes per SM at the sampled SM clock."""
    th = tokens * w.num_kv_heads
    fma = th * ((1 << w.k_bits) + (1 << w.v_bits)) * w.head_dim
    mhz = (clocks or {}).get("sm_mhz") or (clocks or {}).get("sm_max_mhz") or 2070.0
    peak = sms * 128 * mhz * 1e6
    achieved = fma / (ms / 1e3)
    return {"tokens": tokens, "ms": ms, "token_heads_per_s": th / (ms / 1e3),
            "roofline": {"bound": "alu", "achieved": achieved / 1e12, "peak": peak / 1e12,
                         "unit": "TFMA/s", "frac": achieved / peak,
                         "peak_source": f"derived: {sms} SMs x 128 FP32 lanes x {mhz:.0f} MHz",
                         "algorithmic_fma_per_token_head": ((1 << w.k_bits) + (1 << w.v_bits)) * w.head_dim}}


def workload_config(w, splits, copies, balanced=None):
    return {"workload": w.name, "batch": w.batch, "q_heads": w.num_q_heads,
            "kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "context": w.context,
            "attended_tokens_per_step": tokens_per_step(w),
            "k_code": f"d{w.k_sub} x {w.k_bits}-bit", "v_code": f"d{w.v_sub} x {w.v_bits}-bit",
            "page_size": w.page_size, "num_splits": splits,
            "units": None if balanced is None else ("length-balanced" if balanced else "fixed splits"),
            "l2": (f"rotating {copies} cache copies ({copies * code_bytes_per_step(w) / 1e6:.0f} MB"
                   " of codes) > 2x L2" if copies else None)}



# ------------------------------------------------------------- multi-rank ---
# Replicas only: every rank runs the same per-GPU workload with no data-path
# collective; the job's time is the slowest rank's.

def rank_env():
    """(rank, world size, local rank) from the torchrun environment."""
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def max_over_ranks(x, dist, device):
    """The maximum of the per-rank value x over all ranks (x itself without a group)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world, units_per_rank, ms):
    """Whole-job throughput: the units all ranks processed per second of the slowest rank."""
    return world * units_per_rank / (ms / 1e3)

# ----------------------------------------------------------------- our arm ---

def main():
    args = parse()
    rank, world, local = rank_env()
    w = W.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w, rank)
        return

    import torch
    import bit_vector_quantized_gb300 as vq

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if args.methods_only:
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        r = method_comparison(torch, vq, args.workload, dev, 3, l2, measured_hbm()[0], only_launch=True)
        print(json.dumps({"methods_only": w.name, "device_status": r.get("device_status"),
                          "skipped": r.get("skipped")}), flush=True)
        return
    if args.launches_only:
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        r = split_kernel_block(torch, vq, args.workload, dev, 4, l2, measured_hbm()[0],
                               only_launch=True)
        print(json.dumps({"launches_only": w.name, **r}), flush=True)
        assert r["device_status"] == 0, r
        return
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if dist is not None:
            dist.barrier()

    lam, ck, cv = load_calib(args.workload)
    layout = vq.make_layout(w.head_dim, w.num_q_heads, w.num_kv_heads, w.k_sub, w.k_bits,
                            w.v_sub, w.v_bits, w.page_size)
    lens = W.seq_lens(w)
    B = w.batch
    num_pages = W.num_pages(w)
    lam_d = torch.from_numpy(lam).to(dev)
    ck_d = torch.from_numpy(ck).to(dev)
    cv_d = torch.from_numpy(cv).to(dev)
    table_d = torch.from_numpy(W.page_table(w)).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    k_pool, v_pool = vq.alloc_pools(layout, num_pages, dev, zero=True)

    # ---- prefill encode of the cached context (also reported) ----------------
    enc_ms = 0.0
    for b in range(B):
        n = int(lens[b])
        for s0 in range(0, n, 65536):
            s1 = min(n, s0 + 65536)
            kk = torch.from_numpy(W.kv_tokens(w, b, "k", s0, s1)).to(dev)
            vv = torch.from_numpy(W.kv_tokens(w, b, "v", s0, s1)).to(dev)
            sl = torch.from_numpy(W.slot_mapping(w, b, s0, s1)).to(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            vq.encode_kv(layout, kk, vv, sl, lam_d, ck_d, cv_d, k_pool, v_pool, status=status)
            e1.record()
            e1.synchronize()
            enc_ms += e0.elapsed_time(e1)
    prefill_tokens = int(lens.sum())

    # ---- per-step inputs --------------------------------------------------------
    q_h = W.queries(w)
    k_new_h = np.stack([W.kv_tokens(w, b, "k", int(n), int(n) + 1)[0] for b, n in enumerate(lens)])
    v_new_h = np.stack([W.kv_tokens(w, b, "v", int(n), int(n) + 1)[0] for b, n in enumerate(lens)])
    slots_h = np.array([W.slot_mapping(w, b, int(n), int(n) + 1)[0] for b, n in enumerate(lens)])
    q_d = torch.from_numpy(q_h).to(dev)
    k_new = torch.from_numpy(k_new_h).to(dev)
    v_new = torch.from_numpy(v_new_h).to(dev)
    slots_d = torch.from_numpy(slots_h.astype(np.int64)).to(dev)
    seq_d = torch.from_numpy((lens + 1).astype(np.int32)).to(dev)
    max_len = int((lens + 1).max())
    splits = args.splits or vq.vq_default_num_splits(layout, B, max_len)
    ws_bytes = vq.vq_decode_workspace_bytes(layout, B, max_len, splits)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    out = torch.empty((B, w.num_q_heads, w.head_dim), dtype=torch.float16, device=dev)

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    step_bytes = code_bytes_per_step(w)
    copies = args.copies or max(1, -(-2 * l2 // step_bytes))
    pools = [(k_pool, v_pool)] + [(k_pool.clone(), v_pool.clone()) for _ in range(copies - 1)]
    torch.cuda.synchronize()

    def p(t):
        return t.data_ptr()

    def step(i):
        """The hot path: vq_decode_step (append, split attention, merge)."""
        kp, vp = pools[i % copies]
        vq.vq_decode_step(layout, B, p(q_d), p(k_new), p(v_new), p(lam_d), p(ck_d), p(cv_d),
                          p(kp), p(vp), num_pages, p(table_d), table_d.shape[1], p(seq_d), max_len,
                          0.0, splits, p(out), p(ws), ws_bytes, p(status),
                          torch.cuda.current_stream().cuda_stream)

    def step_unfused(i, ev=None):
        """The same step through the separate calls (vq_encode_kv, vq_decode_partial,
        vq_decode_combine), with optional events around each kernel."""
        kp, vp = pools[i % copies]
        stream = torch.cuda.current_stream().cuda_stream
        if ev is not None:
            ev[0].record()
        vq.vq_encode_kv(layout, B, p(k_new), p(v_new), p(slots_d), p(lam_d), p(ck_d), p(cv_d),
                        p(kp), p(vp), num_pages, p(status), stream)
        if ev is not None:
            ev[1].record()
        vq.vq_decode_partial(layout, B, p(q_d), p(lam_d), p(ck_d), p(cv_d), p(kp), p(vp),
                             num_pages, p(table_d), table_d.shape[1], p(seq_d), max_len, 0.0,
                             splits, p(ws), ws_bytes, p(status), stream)
        if ev is not None:
            ev[2].record()
        vq.vq_decode_combine(layout, B, max_len, splits, p(ws), ws_bytes, p(out), stream)
        if ev is not None:
            ev[3].record()

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"

    K = args.steps
    cap = torch.cuda.Stream(device=dev)

    def capture(fn, n):
        gr = torch.cuda.CUDAGraph()
        cap.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(cap):
            with torch.cuda.graph(gr, stream=cap):
                for i in range(n):
                    fn(i)
        torch.cuda.current_stream().wait_stream(cap)
        gr.replay()
        torch.cuda.synchronize()
        return gr

    def split_only(i):
        kp, vp = pools[i % copies]
        vq.vq_decode_partial(layout, B, p(q_d), p(lam_d), p(ck_d), p(cv_d), p(kp), p(vp),
                             num_pages, p(table_d), table_d.shape[1], p(seq_d), max_len, 0.0,
                             splits, p(ws), ws_bytes, p(status), torch.cuda.current_stream().cuda_stream)

    # The timed graph holds the K steps only.  A graph of K back-to-back split
    # launches gives the split kernel's average launch duration for the
    # roofline, and a graph of the steps with event nodes around every kernel
    # gives the per-kernel breakdown (event nodes add their own latency).
    g = capture(step, K)
    g_split = capture(split_only, K)
    n_ev = min(K, 500)
    try:
        evs = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(4)]
               for _ in range(n_ev)]
        g_ev = capture(lambda i: step_unfused(i, evs[i]), n_ev)
        graph_events = True
    except (TypeError, RuntimeError):
        evs, g_ev, graph_events = None, None, False

    # ---- soak (untimed) so clocks settle, then the timed replay ----------------
    sampler = ClockSampler(device_id_for_smi(torch, local))
    t_end = time.time() + args.soak_seconds
    while time.time() < t_end:
        g.replay()
        torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    g.replay()
    t1.record()
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop()
    total_ms = max_over_ranks(t0.elapsed_time(t1), dist, dev)
    ms_per_step = total_ms / K

    if graph_events:
        g_ev.replay()
        torch.cuda.synchronize()
        split_ms = [e[1].elapsed_time(e[2]) for e in evs]
        append_ms = [e[0].elapsed_time(e[1]) for e in evs]
        comb_ms = [e[2].elapsed_time(e[3]) for e in evs]
        timing_note = ("split kernel: a graph of K back-to-back launches between two events; "
                       "breakdown: graph event nodes around each kernel")
    else:  # eager fallback: events around each launch after the timed region
        ev2 = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(min(K, 500))]
        for i, e in enumerate(ev2):
            step_unfused(i, e)
        torch.cuda.synchronize()
        split_ms = [e[1].elapsed_time(e[2]) for e in ev2]
        append_ms = [e[0].elapsed_time(e[1]) for e in ev2]
        comb_ms = [e[2].elapsed_time(e[3]) for e in ev2]
        timing_note = ("split kernel: a graph of K back-to-back launches between two events; "
                       "breakdown: eager launches bracketed by events")
    split_avg = float(np.mean(split_ms))
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    s0.record()
    g_split.replay()
    s1.record()
    torch.cuda.synchronize()
    split_launch_ms = s0.elapsed_time(s1) / K
    assert int(status.item()) == 0, f"device status {int(status.item())}"

    toks = tokens_per_step(w)
    value = job_rate(world, toks, ms_per_step)
    hbm_peak, peak_src = measured_hbm()
    achieved = step_bytes / (split_launch_ms / 1e3) / 1e9
    traffic = recorded_traffic(args.workload)

    # ---- end to end: host buffers, H2D of the step inputs, D2H of the output ---
    e2e = None
    if not args.no_e2e:
        # the step's inputs (q and the new token's K and V) sit back to back in
        # one pinned host buffer and one device buffer, so each step moves
        # them with a single host-to-device copy
        nq, nk = q_h.size, k_new_h.size
        in_p = torch.empty(nq + 2 * nk, dtype=torch.float16).pin_memory()
        in_p[:nq].copy_(torch.from_numpy(q_h).reshape(-1))
        in_p[nq:nq + nk].copy_(torch.from_numpy(k_new_h).reshape(-1))
        in_p[nq + nk:].copy_(torch.from_numpy(v_new_h).reshape(-1))
        in_d = torch.empty(nq + 2 * nk, dtype=torch.float16, device=dev)
        q_e, k_e, v_e = in_d[:nq], in_d[nq:nq + nk], in_d[nq + nk:]
        out_p = torch.empty(out.shape, dtype=out.dtype).pin_memory()

        def e2e_step(i):
            in_d.copy_(in_p, non_blocking=True)
            kp, vp = pools[i % copies]
            vq.vq_decode_step(layout, B, p(q_e), p(k_e), p(v_e), p(lam_d), p(ck_d), p(cv_d),
                              p(kp), p(vp), num_pages, p(table_d), table_d.shape[1], p(seq_d),
                              max_len, 0.0, splits, p(out), p(ws), ws_bytes, p(status),
                              torch.cuda.current_stream().cuda_stream)
            out_p.copy_(out, non_blocking=True)

        # eager: every step pays the Python binding's and the C ABI's host work
        for i in range(3):
            e2e_step(i)
        torch.cuda.synchronize()
        barrier()
        a, bb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for i in range(K):
            e2e_step(i)
        bb.record()
        torch.cuda.synchronize()
        e_ms = max_over_ranks(a.elapsed_time(bb) / K, dist, dev)
        # the same steps replayed from a CUDA graph (host work captured once)
        ge = capture(e2e_step, K)
        barrier()
        a.record()
        ge.replay()
        bb.record()
        torch.cuda.synchronize()
        g_ms = max_over_ranks(a.elapsed_time(bb) / K, dist, dev)
        e2e = {"value": job_rate(world, toks, e_ms), "unit": UNIT,
               "h2d_bytes_per_step": in_p.numel() * 2,
               "d2h_bytes_per_step": out_p.numel() * 2, "ms_per_step": e_ms,
               "how": "eager: per step, one pinned H2D copy of q and the new token's K/V, "
                      "one vq_decode_step call through the Python binding (ctypes -> C ABI), "
                      "D2H of the output; host work included",
               "graph": {"value": job_rate(world, toks, g_ms), "ms_per_step": g_ms,
                         "how": "the same steps captured once in a CUDA graph and replayed"}}

    comparison = unfused = residual = None
    if world == 1 and not args.no_fp16_compare:
        try:
            comparison = fp16_comparison(torch, w, dev, min(K, 200), l2)
            if "us_per_step" in comparison:
                comparison["step_speedup_vs_fp16"] = comparison["us_per_step"] / (1e3 * ms_per_step)
                comparison["attention_speedup_vs_fp16"] = comparison["us_per_step"] / (1e3 * split_launch_ms)
        except Exception as exc:  # context only: never fail the bench line on it
            comparison = {"skipped": f"{type(exc).__name__}: {exc}"[:200]}
        try:
            unfused = unfused_comparison(torch, vq, w, layout, pools, lam_d, ck_d, cv_d, q_d,
                                         num_pages, lens, min(K, 200), dev)
            if "us_per_step" in unfused:
                unfused["step_speedup_vs_unfused"] = unfused["us_per_step"] / (1e3 * ms_per_step)
                unfused["dequantize_hbm_frac"] = unfused["dequantize_gbs"] / hbm_peak
        except Exception as exc:
            unfused = {"skipped": f"{type(exc).__name__}: {exc}"[:200]}
        try:
            residual = residual_comparison(torch, vq, w, layout, pools, lam_d, ck_d, cv_d, q_d,
                                           table_d, seq_d, max_len, num_pages, splits,
                                           min(K, 200), dev)
        except Exception as exc:
            residual = {"skipped": f"{type(exc).__name__}: {exc}"[:200]}

    methods = None
    if world == 1 and not args.no_methods:
        try:
            methods = method_comparison(torch, vq, args.workload, dev, min(K, 200), l2, hbm_peak)
        except Exception as exc:  # context: never fail the bench line on it
            methods = {"skipped": f"{type(exc).__name__}: {exc}"[:200]}

    others = None
    if world == 1 and not args.no_other_workloads:
        others = []
        for wi in (3, 4):
            if wi == args.workload:
                continue
            try:
                others.append(split_kernel_block(torch, vq, wi, dev, min(K, 200), l2, hbm_peak))
            except Exception as exc:  # context: never fail the bench line on it
                others.append({"workload": W.WORKLOADS[wi].name,
                               "skipped": f"{type(exc).__name__}: {exc}"[:200]})

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = run_cpu_baseline(w, lam, ck, cv, args.cpu_seconds)

    if rank == 0:
        cfg = workload_config(w, splits, copies, vq.vq_decode_units_balanced(layout, B, max_len, splits) == 1)
        cfg["parallelism"] = f"replicas x{world}" if world > 1 else "single GPU"
        cfg["graph"] = True
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "fp16 operands (centroids, q~ as fp16 hi+lo, p), fp32 accumulation",
            "data": "synthetic",
            "config": cfg,
            "hbm": {"step_gbs": world * step_bytes / (ms_per_step / 1e3) / 1e9,
                    "split_kernel_gbs": achieved, "pct_of_8tbs_split_kernel": 100 * achieved / NOMINAL_HBM_GBS,
                    "compressed_bytes_per_step": step_bytes},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak, "traffic": traffic,
                         "kernel": "vq_decode_split_kernel", "peak_source": peak_src,
                         "algorithmic_bytes_per_launch": step_bytes, "timing": timing_note},
            "breakdown_us": {"append_encode": 1e3 * float(np.mean(append_ms)),
                             "split_attention": 1e3 * split_avg,
                             "split_attention_back_to_back": 1e3 * split_launch_ms,
                             "combine": 1e3 * float(np.mean(comb_ms)), "step": 1e3 * ms_per_step},
            "prefill_encode": encode_report(w, prefill_tokens, enc_ms, sms, clocks),
            "fp16_comparison": comparison,
            "unfused_comparison": unfused,
            "residual_window": residual,
            "other_workloads": others,
            "methods": methods,
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": step_launches(w, sms) * K,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
