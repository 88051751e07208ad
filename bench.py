"""Benchmark of the DFlash 2 draft cycle on one GB300 (replicas across GPUs).

Headline workload: the full-size drafter (5 layers, width 4096, vocab 151936),
one request, block K=8, 2048 context tokens with a 1024-token window.  One
step = one draft cycle in one CUDA graph: the drafter pass injecting K
target-hidden rows (the most accepted tokens a cycle can add; their K/V formed
inside the pass) + top-16 -> Viterbi selector -> greedy accept.
value = draft cycles per second over all ranks (each GPU runs its own replica).

Also reported: the same cycle with the injection as its own call; the draft
pass alone (draft_block + select_path) at B=1 and at B=32 (ragged contexts in
[512, 8192], paged 64-token pages), each as a fraction of its roofline; the
roofline of the dominant kernel (the tcgen05 projection GEMM) over the pass's
GEMM shapes; the bulk injection of 8 x 4096 rows against the bf16 tensor
roofline; the 4-bit drafter; an end-to-end figure through the C ABI with host
buffers; and the CPU oracle timed on a bounded sample of the same workload.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                  [--only b1,b32,inject,q4 | inject4k | q4lm] [--no-b32] [--no-inject]
                  [--no-cpu-baseline]
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "draft cycles/s (full-size DFlash 2 drafter, B=1, block 8)"
UNIT = "cycles/s"
WORKLOAD = "full drafter: D 4096, 5 layers, 32q/8kv x 128, SwiGLU 14336, vocab 151936; B=1, K=8, context 2048, window 1024, top-16, selector rank 256"


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sus=float(d["bf16_tflops_sustained"]), src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


# ------------------------------------------------------------------ workload shapes

def weight_bytes(cfg):
    es = 2 if cfg["dtype"] == "bf16" else 4
    return {n: int(np.prod(s)) * es for n, s, _ in synth.weight_names(cfg)}


def pass_bytes(cfg, B, K, ctx):
    """Algorithmic bytes of one draft pass (draft_block + select_path): every weight
    the pass multiplies by, once; the window's context K/V; the block's embedding
    rows; the selector's table rows (both projections) of the anchor and the
    candidates."""
    wb = weight_bytes(cfg)
    es = 2
    D, k, r = cfg["d_model"], cfg["top_k"], cfg["sel_rank"]
    w = sum(v for n, v in wb.items()
            if n not in ("fc", "fc_norm", "embed", "sel_pu", "sel_pv", "sel_gate"))
    kv = 0
    per_tok = cfg["n_layers"] * 2 * cfg["n_kv_heads"] * cfg["head_dim"] * es
    for c in ctx:
        kv += min(cfg["window"], int(c)) * per_tok
    gathers = B * K * D * es + B * (1 + (K - 1) * k) * 2 * r * 4
    return w + kv + gathers


def q4_pass_bytes(cfg, B, K, ctx):
    """pass_bytes with the 4-bit matrices counted as their codes (half a byte a
    weight) and (scale, bias) words (4 bytes a row and group of 64)."""
    shapes = {n: s for n, s, _ in synth.weight_names(cfg)}
    out = pass_bytes(cfg, B, K, ctx)
    for n in synth.q4_names(cfg):
        if n == "fc":
            continue  # not read by the pass
        N, Kin = shapes[n]
        out += N * Kin // 2 + N * (Kin // 64) * 4 - N * Kin * 2
    return out


def stored_traffic(n_launches):
    """DRAM bytes (read + write) of one replay of the roofline GEMM sequence, from
    the ncu capture recorded in profiles/ -- only while the library's sources are
    the ones that capture measured (else None)."""
    path = os.path.join(ROOT, "profiles", "gemm_roofline_traffic.json")
    try:
        rec = json.load(open(path))
        from block_diffusion_drafter_inject_gb300.build import source_fingerprint
        if rec.get("source_fingerprint") != source_fingerprint():
            return None
        if rec.get("launches_per_pass") != n_launches:
            return None
        return rec["dram_bytes_per_pass"]
    except (OSError, ValueError, KeyError):
        return None


def pass_gemms(cfg, B, K):
    """(N_out, K_in, T, weight name) of every projection GEMM of one draft pass.
    At 16 block rows or fewer (bf16) the conv gate linears run inside the fused
    conv kernels, not as GEMMs; the selector reads its prepared table (no
    projection GEMMs per pass)."""
    D, F, V = cfg["d_model"], cfg["d_ff"], cfg["vocab"]
    Hq, Hkv, dh = cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"]
    GW = 2 * D // cfg["conv_group"]
    T = B * K
    gates = not (cfg["dtype"] == "bf16" and T <= 16)
    out = []
    for l in range(cfg["n_layers"]):
        p = f"layers.{l}."
        g = [(GW, D, T, p + f"conv_w.{i}") for i in range(4)] if gates else [None] * 4
        out += [g[0], ((Hq + 2 * Hkv) * dh, D, T, p + "wqkv"), (D, Hq * dh, T, p + "wo"), g[1],
                g[2], (2 * F, D, T, p + "w_gate_up"), (D, F, T, p + "w_down"), g[3]]
    out = [x for x in out if x is not None]
    out.append((V, D, B * (K - 1), "lm_head"))
    return out


def window_layout(ctx, K, P, W, seed):
    """Page table holding only the pages a pass touches: positions [ctx-W, ctx+K)."""
    B = len(ctx)
    maxp = max((int(c) + K + P - 1) // P for c in ctx)
    need = []
    for c in ctx:
        lo = max(0, int(c) - W)
        need.append(list(range(lo // P, (int(c) + K - 1) // P + 1)))
    total = sum(len(n) for n in need)
    perm = synth.stream(seed, "page_perm").permutation(total)
    table = np.full((B, maxp), -1, dtype=np.int32)
    o = 0
    for b, pages in enumerate(need):
        for pi in pages:
            table[b, pi] = perm[o]
            o += 1
    return table, total


# ------------------------------------------------------------------ clocks

class Clocks:
    """nvidia-smi clock and throttle-reason samples (every 200 ms) while the
    block runs, kept in a temporary file that is removed afterwards."""

    def __init__(self):
        self.proc = None
        fd, self.path = tempfile.mkstemp(prefix="dflash_clocks_", suffix=".csv")
        os.close(fd)

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=index,clocks.sm,clocks.max.sm,power.draw,"
                 "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
                 "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                 "clocks_event_reasons.sw_power_cap", "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self._stop()
        try:
            os.remove(self.path)
        except OSError:
            pass

    def _stop(self):
        if self.proc and self.proc.poll() is None:
            self.proc.terminate()
            try:
                self.proc.wait(5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self, gpu_index):
        """Median SM clock, max clock and throttle reasons seen so far (stops sampling)."""
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self._stop()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9 or f[0] != str(gpu_index):
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------------------ GPU arm

def event_time(torch, fn, steps, warmup, barrier=None):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    if barrier:
        barrier()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(steps):
        fn()
    e.record()
    torch.cuda.synchronize()
    if barrier:
        barrier()
    return s.elapsed_time(e) / steps   # ms per step


def capture(torch, fn):
    fn()                                   # first call sets kernel attributes
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def setup_workload(torch, dfl, cfg, Wd, B, K, ctx, seed, max_inject):
    """Paged KV holding the injected window of every request; device inputs of a cycle."""
    P, Wn = cfg["page_size"], cfg["window"]
    table, npages = window_layout(ctx, K, P, Wn, seed)
    kv = dfl.PagedKV(cfg, table, npages, "cuda")
    cyc = dfl.DraftCycle(cfg, Wd, kv, B, K, max_inject, "cuda")
    # prefill: inject each request's window (synthetic hidden states), in chunks
    req = np.concatenate([np.full(min(Wn, int(c)), b, np.int32) for b, c in enumerate(ctx)])
    pos = np.concatenate([np.arange(max(0, int(c) - Wn), int(c), dtype=np.int32) for c in ctx])
    hid = synth.make_hiddens(cfg, len(req), seed=seed, name="prefill_hiddens")
    for o in range(0, len(req), max_inject):
        sl = slice(o, o + max_inject)
        dfl.inject_context(cfg, Wd, kv, torch.from_numpy(hid[sl]).to(torch.bfloat16).cuda(),
                           torch.from_numpy(req[sl]).cuda(), torch.from_numpy(pos[sl]).cuda(),
                           cyc.ws)
    torch.cuda.synchronize()
    # per-cycle inputs: re-inject the last K context rows of every request
    creq = np.repeat(np.arange(B, dtype=np.int32), K)
    cpos = np.concatenate([np.arange(int(c) - K, int(c), dtype=np.int32) for c in ctx])
    ch = synth.make_hiddens(cfg, B * K, seed=seed, name="cycle_hiddens")
    inp = dict(
        hidden=torch.from_numpy(ch).to(torch.bfloat16).cuda(),
        req=torch.from_numpy(creq).cuda(), pos=torch.from_numpy(cpos).cuda(),
        anchor=torch.from_numpy(synth.make_anchors(cfg, B, seed=seed)).cuda(),
        ctx=torch.from_numpy(np.asarray(ctx, np.int32)).cuda(),
        target=torch.from_numpy(synth.make_target_logits(cfg, B, K, seed=seed)).cuda())
    return kv, cyc, inp


def inject_weight_names(cfg):
    """The weights an inject call reads: fc and its norm, every layer's wqkv and k_norm."""
    names = {"fc_norm", "fc"}
    for l in range(cfg["n_layers"]):
        names |= {f"layers.{l}.wqkv", f"layers.{l}.k_norm"}
    return names


def bench_inject_rows(torch, dfl, cfg, pk, args, N=4096):
    """One inject call of N rows into one request's pages, with only the weights
    injection reads on the device (about 1.2 GB in all): the small case on which
    the injection's GEMMs are profiled."""
    Wh = synth.make_weights(cfg, seed=0, names=inject_weight_names(cfg))
    Wd = dfl.DeviceWeights.from_host(cfg, Wh, "cuda")
    P = cfg["page_size"]
    kv = dfl.PagedKV(cfg, np.arange(N // P, dtype=np.int32)[None, :], N // P, "cuda")
    ws = dfl.Workspace(cfg, 1, 2, N)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(3)
    hid = torch.randn((N, cfg["n_taps"] * cfg["d_target"]), device="cuda",
                      generator=gen).to(torch.bfloat16)
    req = torch.zeros(N, dtype=torch.int32, device="cuda")
    pos = torch.arange(N, dtype=torch.int32, device="cuda")

    def inject():
        dfl.inject_context(cfg, Wd, kv, hid, req, pos, ws)

    steps = max(3, min(args.steps, 20))
    ms = event_time(torch, inject, steps, args.warmup)
    fl = inject_flops(cfg, N)
    return {"rows": N, "inject_ms": ms, "inject_tflops": fl / (ms * 1e-3) / 1e12,
            "frac_of_tensor_roofline": fl / (pk["bf16_sus"] * 1e12) / (ms * 1e-3),
            "device_status": dfl.read_device_status(ws)}


def bench_q4_lm_head(torch, dfl, cfg, pk, args, T=7):
    """The 4-bit lm_head GEMM alone (vocab x d_model, T tokens) with only its records
    on the device (350 MB of random bytes: the time does not depend on the values):
    the small case on which the 4-bit GEMM is profiled."""
    V, D = cfg["vocab"], cfg["d_model"]
    nbytes = (V + 127) // 128 * 2 * (D // 64) * 2304
    gen = torch.Generator(device="cuda")
    gen.manual_seed(4)
    rec = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device="cuda", generator=gen)
    X = torch.randn((T, D), device="cuda", generator=gen).to(torch.bfloat16)
    S = dfl.linear_splits(V, T, D)
    out = torch.empty((S, T, V), device="cuda", dtype=torch.float32)
    steps = max(3, min(args.steps, 20))
    ms = event_time(torch, lambda: dfl.linear_q4(rec, V, X, out, S), steps, args.warmup)
    return {"shape": [V, D, T], "us": ms * 1e3, "record_bytes": nbytes,
            "gbs": nbytes / (ms * 1e-3) / 1e9, "frac_of_hbm": nbytes / (ms * 1e-3) / 1e9 / pk["hbm"]}


def run_gpu(args, rank, world, barrier, allmax):
    import torch
    import block_diffusion_drafter_inject_gb300 as dfl

    dev = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(dev)
    cfg = synth.preset("full")
    pk = peaks()
    if args.sections == {"inject4k"}:
        return {"inject4k": bench_inject_rows(torch, dfl, cfg, pk, args)}, None
    if args.sections == {"q4lm"}:
        return {"q4lm": bench_q4_lm_head(torch, dfl, cfg, pk, args)}, None
    t0 = time.time()
    Wh = synth.make_weights(cfg, seed=0)
    Wd = dfl.DeviceWeights.from_host(cfg, Wh, "cuda")
    # the selector's projections of every vocabulary row, formed once per weight set
    tab_ws = dfl.Workspace(cfg, 1, 2, 1)
    dfl.prepare_selector(cfg, Wd, tab_ws)
    torch.cuda.synchronize()
    del tab_ws
    res = {"gpu": torch.cuda.get_device_name(dev), "setup_s": round(time.time() - t0, 1)}
    sections = args.sections
    if "b1" in sections:
        res.update(bench_b1(torch, dfl, cfg, Wd, pk, args, world, barrier, allmax, dev))
    if "b32" in sections:
        res["b32"] = bench_b32(torch, dfl, cfg, Wd, pk, args)
    if "inject" in sections:
        res["inject"] = bench_inject(torch, dfl, cfg, Wd, pk, args)
    if "q4" in sections:
        res["q4"] = bench_q4(torch, dfl, cfg, Wh, pk, args)
    return res, Wh


def headline_config(cfg, world):
    """The `config` of the headline line, shared by both arms."""
    return {"workload": WORKLOAD, "B": 1, "K": 8, "ctx": 2048, "window": cfg["window"],
            "cycle": "draft_block_inject (K new context rows injected inside the pass) + "
                     "select_path + accept_greedy, one CUDA graph",
            "l2": "inputs larger than L2: 3.5 GB of weights streamed per step, no flush",
            "parallelism": f"replicas x{world}"}


def bench_b1(torch, dfl, cfg, Wd, pk, args, world, barrier, allmax, dev):
    """The headline: one draft cycle at B=1, K=8, context 2048 (one CUDA graph)."""
    B, K, ctx = 1, 8, [2048]
    kv, cyc, inp = setup_workload(torch, dfl, cfg, Wd, B, K, ctx, 0, 1024)

    def cycle():
        cyc.run(inp["hidden"], inp["req"], inp["pos"], inp["anchor"], inp["ctx"], inp["target"])

    def cycle_two_calls():
        cyc.run(inp["hidden"], inp["req"], inp["pos"], inp["anchor"], inp["ctx"], inp["target"],
                fused=False)

    def dpass():
        dfl.draft_block(cfg, Wd, kv, inp["anchor"], inp["ctx"], K, cyc.ws, cyc.topk_ids,
                        cyc.topk_logp)
        dfl.select_path(cfg, Wd, inp["anchor"], cyc.topk_ids, cyc.topk_logp, K, cyc.ws, cyc.path,
                        cyc.score)

    dfl.launch_count(reset=True)
    cycle()
    torch.cuda.synchronize()
    launches_per_cycle = dfl.launch_count(reset=True)
    status = dfl.read_device_status(cyc.ws)
    g_cycle = capture(torch, cycle)
    g_two = capture(torch, cycle_two_calls)
    g_pass = capture(torch, dpass)

    with Clocks() as clk:
        torch.cuda.nvtx.range_push("b1_cycle")  # lets a profiler select these launches
        ms_cycle = event_time(torch, g_cycle.replay, args.steps, args.warmup, barrier)
        torch.cuda.nvtx.range_pop()
        torch.cuda.nvtx.range_push("b1_pass")  # lets a profiler select these launches
        ms_pass = event_time(torch, g_pass.replay, args.steps, args.warmup)
        torch.cuda.nvtx.range_pop()
        ms_two = event_time(torch, g_two.replay, args.steps, args.warmup)
        clocks = clk.summary(dev)
    ms_cycle = allmax(ms_cycle)

    # ---------------- dominant kernel: the projection GEMM at the pass's shapes
    gem = pass_gemms(cfg, B, K)
    xs = {}
    outs = {}
    gem_bytes = 0
    for (N, Kin, T, name) in gem:
        key = (T, Kin)
        if key not in xs:
            xs[key] = torch.randn((T, Kin), device="cuda").to(torch.bfloat16)
        S = dfl.linear_splits(N, T, Kin)
        outs[(N, Kin, T)] = (torch.empty((S, T, N), device="cuda", dtype=torch.float32), S)
        gem_bytes += N * Kin * 2 + T * Kin * 2 + T * N * 4

    def gemms():
        for (N, Kin, T, name) in gem:
            o, S = outs[(N, Kin, T)]
            dfl.linear(Wd.t[name], xs[(T, Kin)], o, S)

    g_gemm = capture(torch, gemms)
    torch.cuda.nvtx.range_push("gemm_roofline")  # lets a profiler select these launches
    ms_gemm = event_time(torch, g_gemm.replay, args.steps, args.warmup)
    torch.cuda.nvtx.range_pop()
    gemm_gbs = gem_bytes / (ms_gemm * 1e-3) / 1e9
    traffic = stored_traffic(len(gem))

    # ---------------- e2e through the C ABI with host buffers
    # The step's inputs other than the target logits (hidden rows, request and
    # position ids, anchor, context lengths) sit in one pinned host buffer and one
    # device buffer, each at a 256-byte offset, so that they cross in one copy; the
    # results (accept_len, tokens) likewise come back in one.
    names = [k for k in inp if k != "target"]
    offs, size = {}, 0
    for k in names:
        offs[k] = size
        size += (inp[k].numel() * inp[k].element_size() + 255) // 256 * 256

    def views(buf):
        return {k: buf[offs[k]:offs[k] + inp[k].numel() * inp[k].element_size()]
                .view(inp[k].dtype).view(inp[k].shape) for k in names}

    dev_pack = torch.empty(size, dtype=torch.uint8, device="cuda")
    host_pack = torch.empty(size, dtype=torch.uint8).pin_memory()
    dinp, hinp = views(dev_pack), views(host_pack)
    for k in names:
        dinp[k].copy_(inp[k])
        hinp[k].copy_(inp[k].cpu())
    dinp["target"] = inp["target"]
    pin_target = inp["target"].cpu().pin_memory()
    dev_out = torch.empty(B + B * K, dtype=torch.int32, device="cuda")
    host_out = torch.empty(B + B * K, dtype=torch.int32).pin_memory()
    d_acc, d_tok = dev_out[:B], dev_out[B:].view(B, K)
    h2d = size + pin_target.numel() * pin_target.element_size()
    d2h = host_out.numel() * 4

    # The target's logits are read only by acceptance: the serving loop copies them
    # on a side stream while the pass runs (once the previous step's acceptance has
    # been issued, so that the buffer it reads is not overwritten); the rest of the
    # inputs go first on the main stream.
    def front():
        dfl.draft_block_inject(cfg, Wd, kv, dinp["hidden"], dinp["req"], dinp["pos"],
                               dinp["anchor"], dinp["ctx"], K, cyc.ws, cyc.topk_ids,
                               cyc.topk_logp)
        dfl.select_path(cfg, Wd, dinp["anchor"], cyc.topk_ids, cyc.topk_logp, K, cyc.ws, cyc.path,
                        cyc.score)

    def back():
        dfl.accept_greedy(cyc.path, dinp["target"], cyc.ws, d_acc, d_tok)

    g_front = capture(torch, front)
    g_back = capture(torch, back)
    side = torch.cuda.Stream()
    ev_free, ev_copied = torch.cuda.Event(), torch.cuda.Event()

    def e2e_step():
        main = torch.cuda.current_stream()
        dev_pack.copy_(host_pack, non_blocking=True)
        ev_free.record(main)
        side.wait_event(ev_free)
        with torch.cuda.stream(side):
            dinp["target"].copy_(pin_target, non_blocking=True)
            ev_copied.record(side)
        g_front.replay()
        main.wait_event(ev_copied)
        g_back.replay()
        host_out.copy_(dev_out, non_blocking=True)

    ms_e2e = allmax(event_time(torch, e2e_step, args.steps, args.warmup, barrier))
    torch.cuda.synchronize()
    # the packed copies carry the same step as the device-resident cycle
    e2e_same = bool(torch.equal(host_out[:B], cyc.accept_len.cpu()) and
                    torch.equal(host_out[B:], cyc.tokens.cpu().view(-1)))

    pb1 = pass_bytes(cfg, B, K, ctx)
    return {
        "metric": METRIC, "value": whole_job_value(world, ms_cycle), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_cycle,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,0.02) weights, N(0,1) target hiddens, N(0,3) target logits)",
        "config": headline_config(cfg, world),
        "draft_pass_us": ms_pass * 1e3,
        "cycle_two_calls_us": ms_two * 1e3,
        "draft_pass_bytes": pb1,
        "draft_pass_hbm_frac": pb1 / (ms_pass * 1e-3) / 1e9 / pk["hbm"],
        "roofline": {"kernel": "k_gemm_tc (tcgen05 projection GEMM, all shapes of one B=1 pass)",
                     "bound": "hbm", "achieved": gemm_gbs, "peak": pk["hbm"], "unit": "GB/s",
                     "frac": gemm_gbs / pk["hbm"], "traffic": traffic,
                     "algorithmic_bytes_per_pass": gem_bytes, "us_per_pass": ms_gemm * 1e3,
                     "peak_source": pk["src"]},
        "e2e": {"value": whole_job_value(world, ms_e2e), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "note": "target logits copied on a side stream during the pass, joined before "
                        "acceptance; the other inputs in one packed copy before the pass, the "
                        "results in one copy after it",
                "result_matches_device_cycle": e2e_same},
        "gpu_launches": launches_per_cycle * args.steps,
        "launches_per_cycle": launches_per_cycle,
        "clocks": clocks,
        "device_status": status,
    }


def bench_b32(torch, dfl, cfg, Wd, pk, args):
    """The draft pass and cycle at B=32 (ragged contexts in [512, 8192], paged)."""
    B2, K = 32, 8
    ctx2 = synth.make_ctx_lens(B2, 512, 8192, seed=1).tolist()
    kv2, cyc2, inp2 = setup_workload(torch, dfl, cfg, Wd, B2, K, ctx2, 1, 4096)

    def dpass2():
        dfl.draft_block(cfg, Wd, kv2, inp2["anchor"], inp2["ctx"], K, cyc2.ws, cyc2.topk_ids,
                        cyc2.topk_logp)
        dfl.select_path(cfg, Wd, inp2["anchor"], cyc2.topk_ids, cyc2.topk_logp, K, cyc2.ws,
                        cyc2.path, cyc2.score)

    def cycle2(fused=True):
        cyc2.run(inp2["hidden"], inp2["req"], inp2["pos"], inp2["anchor"], inp2["ctx"],
                 inp2["target"], fused=fused)

    gp2 = capture(torch, dpass2)
    gc2 = capture(torch, cycle2)
    gt2 = capture(torch, lambda: cycle2(False))
    torch.cuda.nvtx.range_push("b32_pass")  # lets a profiler select these launches
    ms_p2 = event_time(torch, gp2.replay, max(5, args.steps // 2), args.warmup)
    torch.cuda.nvtx.range_pop()
    ms_c2 = event_time(torch, gc2.replay, max(5, args.steps // 2), args.warmup)
    ms_t2 = event_time(torch, gt2.replay, max(5, args.steps // 2), args.warmup)
    status = dfl.read_device_status(cyc2.ws)
    pb2 = pass_bytes(cfg, B2, K, ctx2)
    fl2 = sum(2.0 * N * Kin * T for (N, Kin, T, _) in pass_gemms(cfg, B2, K))
    t_hbm = pb2 / (pk["hbm"] * 1e9)
    t_tc = fl2 / (pk["bf16_sus"] * 1e12)
    return {"draft_pass_us": ms_p2 * 1e3, "cycle_us": ms_c2 * 1e3,
            "cycle_two_calls_us": ms_t2 * 1e3,
            "cycles_per_s": 1e3 / ms_c2, "pass_bytes": pb2, "pass_gemm_flops": fl2,
            "hbm_floor_us": t_hbm * 1e6, "tensor_floor_us": t_tc * 1e6,
            "frac_of_tighter_roofline": max(t_hbm, t_tc) / (ms_p2 * 1e-3),
            "ctx_range": [min(ctx2), max(ctx2)], "device_status": status}


def bench_q4(torch, dfl, cfg, Wh, pk, args):
    """The headline workload (B=1, block 8, context 2048) with the 4-bit drafter:
    fc, QKV, O, gate/up, down and lm_head as 4-bit codes with a (scale, bias) per
    row and 64 input features (seeded synthetic codes)."""
    B, K, ctx = 1, 8, [2048]
    cq = dict(cfg, weight_bits=4)
    Q = synth.make_q4_weights(cq, seed=0)
    Wq = dfl.DeviceWeights.from_host(cq, Wh, "cuda", q4=Q)
    del Q
    tab_ws = dfl.Workspace(cq, 1, 2, 1)
    dfl.prepare_selector(cq, Wq, tab_ws)
    kv, cyc, inp = setup_workload(torch, dfl, cq, Wq, B, K, ctx, 0, 1024)

    def cycle():
        cyc.run(inp["hidden"], inp["req"], inp["pos"], inp["anchor"], inp["ctx"], inp["target"])

    def dpass():
        dfl.draft_block(cq, Wq, kv, inp["anchor"], inp["ctx"], K, cyc.ws, cyc.topk_ids,
                        cyc.topk_logp)
        dfl.select_path(cq, Wq, inp["anchor"], cyc.topk_ids, cyc.topk_logp, K, cyc.ws, cyc.path,
                        cyc.score)

    g_cycle = capture(torch, cycle)
    g_pass = capture(torch, dpass)
    torch.cuda.nvtx.range_push("q4_cycle")  # lets a profiler select these launches
    ms_cycle = event_time(torch, g_cycle.replay, args.steps, args.warmup)
    torch.cuda.nvtx.range_pop()
    torch.cuda.nvtx.range_push("q4_pass")
    ms_pass = event_time(torch, g_pass.replay, args.steps, args.warmup)
    torch.cuda.nvtx.range_pop()
    status = dfl.read_device_status(cyc.ws)
    # the 4-bit GEMMs of one pass replayed back to back
    gem = [(N, Kin, T, n) for (N, Kin, T, n) in pass_gemms(cq, B, K)
           if n.split(".")[-1] in ("wqkv", "wo", "w_gate_up", "w_down", "lm_head")]
    xs, outs, gbytes = {}, {}, 0
    for (N, Kin, T, n) in gem:
        if (T, Kin) not in xs:
            xs[(T, Kin)] = torch.randn((T, Kin), device="cuda").to(torch.bfloat16)
        S = dfl.linear_splits(N, T, Kin)
        while (Kin // 64) % S:
            S -= 1
        outs[n] = (torch.empty((S, T, N), device="cuda", dtype=torch.float32), S)
        gbytes += (N + 127) // 128 * 128 * (Kin // 64) * 2304 // 64 + T * Kin * 2 + S * T * N * 4

    def gemms():
        for (N, Kin, T, n) in gem:
            o, S = outs[n]
            dfl.linear_q4(Wq.t[n + ".q4"], N, xs[(T, Kin)], o, S)

    g_gemm = capture(torch, gemms)
    torch.cuda.nvtx.range_push("q4_gemm_roofline")
    ms_gemm = event_time(torch, g_gemm.replay, args.steps, args.warmup)
    torch.cuda.nvtx.range_pop()
    pb = q4_pass_bytes(cq, B, K, ctx)
    del g_cycle, g_pass, g_gemm
    return {"workload": "B=1, block 8, context 2048, 4-bit fc/QKV/O/gate-up/down/lm_head "
                        "(codes + bf16 scale and bias per 64 inputs)",
            "cycle_us": ms_cycle * 1e3, "cycles_per_s": 1e3 / ms_cycle,
            "draft_pass_us": ms_pass * 1e3, "draft_pass_bytes": pb,
            "draft_pass_hbm_frac": pb / (ms_pass * 1e-3) / 1e9 / pk["hbm"],
            "gemm": {"kernel": "k_gemm_q4 (4-bit weights, tcgen05), the pass's 21 shapes",
                     "bytes_per_pass": gbytes, "us_per_pass": ms_gemm * 1e3,
                     "achieved_gbs": gbytes / (ms_gemm * 1e-3) / 1e9,
                     "frac_of_hbm": gbytes / (ms_gemm * 1e-3) / 1e9 / pk["hbm"]},
            "device_status": status}


def inject_flops(cfg, N):
    """Multiply-add flops of injecting N target-hidden rows: the fc projection and
    every layer's K and V projections."""
    D, Hkv, dh = cfg["d_model"], cfg["n_kv_heads"], cfg["head_dim"]
    TIN = cfg["n_taps"] * cfg["d_target"]
    return 2.0 * N * (D * TIN + cfg["n_layers"] * 2 * Hkv * dh * D)


def bench_inject(torch, dfl, cfg, Wd, pk, args):
    """Context capture at scale: 8 requests each inject 4096 new target-hidden rows
    (5 x 5120 bf16) into their paged draft KV in one call, then one block-16 draft
    cycle runs for all 8 requests."""
    B, K, n = 8, 16, 4096
    N = B * n
    P = cfg["page_size"]
    TIN = cfg["n_taps"] * cfg["d_target"]
    per = (n + K + P - 1) // P
    table = np.arange(B * per, dtype=np.int32).reshape(B, per)
    perm = synth.stream(5, "inject_page_perm").permutation(B * per).astype(np.int32)
    table = perm[table]
    kv = dfl.PagedKV(cfg, table, B * per, "cuda")
    cyc = dfl.DraftCycle(cfg, Wd, kv, B, K, N, "cuda")
    gen = torch.Generator(device="cuda")
    gen.manual_seed(5)
    hid = torch.randn((N, TIN), device="cuda", generator=gen).to(torch.bfloat16)
    req = torch.arange(B, dtype=torch.int32, device="cuda").repeat_interleave(n)
    pos = torch.arange(n, dtype=torch.int32, device="cuda").repeat(B)
    anchor = torch.from_numpy(synth.make_anchors(cfg, B, seed=5)).cuda()
    ctx = torch.full((B,), n, dtype=torch.int32, device="cuda")
    target = torch.from_numpy(synth.make_target_logits(cfg, B, K, seed=5)).cuda()

    def inject():
        dfl.inject_context(cfg, Wd, kv, hid, req, pos, cyc.ws)

    def cycle():
        cyc.run(None, None, None, anchor, ctx, target)

    g_inj = capture(torch, inject)
    g_cyc = capture(torch, cycle)
    steps = max(3, min(args.steps, 20))
    # the cycle is timed first, on the context one injection wrote: timed after the
    # injection's replays it would inherit the clock that seconds of tensor-bound
    # work leave behind (it moved by ~10 % with the injection's own speed)
    g_inj.replay()
    torch.cuda.synchronize()
    ms_cyc = event_time(torch, g_cyc.replay, max(5, args.steps // 2), args.warmup)
    torch.cuda.nvtx.range_push("inject_32k")  # lets a profiler select these launches
    ms_inj = event_time(torch, g_inj.replay, steps, args.warmup)
    torch.cuda.nvtx.range_pop()
    status = dfl.read_device_status(cyc.ws)
    fl = inject_flops(cfg, N)
    t_tc = fl / (pk["bf16_sus"] * 1e12)
    cb = pass_bytes(cfg, B, K, [n] * B)
    return {"workload": f"{B} requests x {n} injected rows ({cfg['n_taps']} x {cfg['d_target']} "
                        f"bf16), then one block-{K} cycle for all {B}",
            "rows": N, "inject_ms": ms_inj, "inject_tflops": fl / (ms_inj * 1e-3) / 1e12,
            "inject_flops": fl, "tensor_floor_ms": t_tc * 1e3,
            "frac_of_tensor_roofline": t_tc / (ms_inj * 1e-3), "peak_tflops": pk["bf16_sus"],
            "peak_kind": "bf16 sustained (measured)",
            "cycle_us": ms_cyc * 1e3, "cycle_pass_bytes": cb,
            "cycle_hbm_frac": cb / (ms_cyc * 1e-3) / 1e9 / pk["hbm"], "device_status": status}


# ------------------------------------------------------------------ CPU oracle

def oracle_sample(cfg, Wh, K=8, ctx=2048, reps=1, seed=0):
    """Time the unmodified oracle on a bounded sample of the headline cycle: layer 0
    of the drafter, 1/L of the lm_head's vocabulary rows, the per-cycle injection
    through that layer, the selector and greedy accept.  Returns (seconds per
    sample, fraction of one cycle's weight parameters the sample touches)."""
    import oracle
    L = cfg["n_layers"]
    Vs = cfg["vocab"] // L
    scfg = dict(cfg, n_layers=1, vocab=Vs, mask_token_id=Vs - 1)
    Ws = {k: v for k, v in Wh.items() if not k.startswith("layers.") or k.startswith("layers.0.")}
    Ws["lm_head"] = Wh["lm_head"][:Vs]
    g = synth.stream(seed, "oracle_ctx")
    n = min(ctx, cfg["window"])
    shape = (ctx, cfg["n_kv_heads"], cfg["head_dim"])
    ck = np.zeros(shape, np.float32)
    cv = np.zeros(shape, np.float32)
    ck[ctx - n:] = g.standard_normal((n,) + shape[1:], dtype=np.float32)
    cv[ctx - n:] = g.standard_normal((n,) + shape[1:], dtype=np.float32)
    hid = synth.make_hiddens(cfg, K, seed=seed, name="cycle_hiddens")
    anchor = synth.make_anchors(scfg, 1, seed=seed)
    target = synth.make_target_logits(cfg, 1, K, seed=seed)
    times = []
    for _ in range(reps):
        t = time.perf_counter()
        oracle.inject_context(scfg, Ws, hid, np.arange(ctx - K, ctx), "bf16")
        d = oracle.draft_block(scfg, Ws, [[ck]], [[cv]], anchor, [ctx], K, "bf16")
        path, _ = oracle.select_path(scfg, Ws, anchor, d["ids"], d["logp"])
        oracle.accept_greedy(path, target)
        times.append(time.perf_counter() - t)
    full = sum(int(np.prod(s)) for n, s, _ in synth.weight_names(cfg) if n not in ("embed", "sel_gate"))
    samp = sum(int(np.prod(s)) for n, s, _ in synth.weight_names(scfg) if n not in ("embed", "sel_gate"))
    return float(np.median(times)), samp / full


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def cpu_baseline(Wh, cfg):
    t, frac = oracle_sample(cfg, Wh, reps=3)
    return {"value": frac / t, "unit": UNIT, "cores": cores(), "kind": "oracle",
            "sample": f"oracle (NumPy float64) on layer 0 + 1/{cfg['n_layers']} of the lm_head rows "
                      f"+ per-cycle inject + selector + accept of the B=1 K=8 cycle; "
                      f"{t:.2f} s per sample (median of 3), sample = {frac:.3f} of the cycle's "
                      f"weight parameters, value = fraction / seconds"}


def run_reference(args):
    """The oracle as it stands on the host cores, on this workload's metric."""
    cfg = synth.preset("full")
    Wh = synth.make_weights(cfg, seed=0)
    for _ in range(args.warmup):
        oracle_sample(cfg, Wh, reps=1)
    ts, frac = [], None
    t0 = time.perf_counter()
    for _ in range(args.steps):
        t, frac = oracle_sample(cfg, Wh, reps=1)
        ts.append(t)
    total = time.perf_counter() - t0
    sec_per_cycle = (total / args.steps) / frac
    v = 1.0 / sec_per_cycle
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": headline_config(cfg, int(os.environ.get("WORLD_SIZE", "1"))),
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores(), "kind": "oracle",
                             "sample": f"each step: oracle on layer 0 + 1/5 of lm_head rows + "
                                       f"inject + select + accept = {frac:.3f} of a cycle's weights"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ------------------------------------------------------------------ replicas

def replica_sync(world, device="cuda"):
    """(barrier, allmax) over the ranks of an already-initialised process group.

    Replicas share nothing on the data path: the only cross-rank traffic is
    the barrier around the timed region and the max of the per-rank step
    times (whole-job throughput = ranks x steps / slowest rank's time)."""
    if world <= 1:
        return None, (lambda x: x)
    import torch
    import torch.distributed as dist
    if not dist.is_initialized():
        if device == "cuda":
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl" if device == "cuda" else "gloo")

    def barrier():
        dist.barrier()

    def allmax(x):
        t = torch.tensor([float(x)], dtype=torch.float64,
                         device=device if device == "cuda" else "cpu")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    return barrier, allmax


def whole_job_value(world, ms_per_step_max):
    """Cycles per second over all replicas for the slowest rank's step time."""
    return world * 1e3 / ms_per_step_max


# ------------------------------------------------------------------ main

def spawn_replicas(n, argv):
    """Re-run this script under torch.distributed.run with n ranks on this node (one
    replica per GPU) and return its exit status; rank 0 prints the JSON line."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node",
           str(n), "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.abspath(__file__)] + list(argv)
    return subprocess.call(cmd)


def replica_selftest(world, rank):
    """CPU check of the replica plumbing (gloo): every rank joins, passes the
    barrier and agrees on the max of the per-rank step times."""
    barrier, allmax = replica_sync(world, device="cpu")
    if barrier:
        barrier()
    worst = allmax(float(rank + 1))
    if rank == 0:
        print(json.dumps({"replica_selftest": True, "world": world, "max_step": worst,
                          "value": whole_job_value(world, worst)}))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--only", default="",
                    help="comma list of sections to run: b1 (headline), b32, inject, q4 "
                         "(the headline workload with 4-bit weights); or, alone, a small "
                         "profiling case: inject4k (a 4096-row injection with only its weights "
                         "loaded) or q4lm (the 4-bit lm_head GEMM with only its records)")
    ap.add_argument("--no-b32", action="store_true")
    ap.add_argument("--no-inject", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--replica-selftest", action="store_true",
                    help="check the replica barrier / max on CPU (gloo) and exit")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    args.sections = set(x for x in args.only.split(",") if x) or {"b1", "b32", "inject", "q4"}
    if args.no_b32:
        args.sections.discard("b32")
    if args.no_inject:
        args.sections.discard("inject")

    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        sys.exit(spawn_replicas(args.gpus, sys.argv[1:]))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))

    if args.replica_selftest:
        replica_selftest(world, rank)
        return

    if args.impl == "reference":
        if rank == 0:
            args.steps = max(1, min(args.steps, 20))  # ~1.4 s of host work per step
            args.warmup = 3
            print(json.dumps(run_reference(args)))
        return

    barrier, allmax = replica_sync(world, device="cuda")
    res, Wh = run_gpu(args, rank, world, barrier, allmax)
    if rank == 0:
        if not args.no_cpu_baseline and "b1" in args.sections and Wh is not None:
            res["cpu_baseline"] = cpu_baseline(Wh, synth.preset("full"))
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
