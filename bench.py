"""Benchmark: one layer-sliding fine-tuning step of the 8B-shape GQA decoder
(32 layers, hidden 4096, 32/8 heads x 128, SwiGLU 14336, vocab 128256,
batch 8 x seq 2048, bf16 weights streamed from pinned host memory through a
3-slot GPU ring, host Adam on fp32 masters) on one GB300.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config 8b] [--impl ours|reference]

Prints one JSON line.  value = tokens/s over K steps timed with CUDA events
(device clock; every step's host Adam update, the last one's included, lies
inside the timed region); e2e = the same through the public
call with host wall clock, including the per-step staging of the token batch
and the read of the loss.  --impl reference times the CPU oracle on a bounded
sample of the same workload.

The library drives one GPU: its GEMM clusters share weight tiles by TMA
multicast within that GPU's own memory, and the step has no cross-GPU
exchange.  A launch on more than one GPU (--gpus N > 1, or WORLD_SIZE > 1
under torchrun) is refused: rank 0 prints one JSON line with an
"unavailable" reason and every rank exits 0 without touching a GPU.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import inputs  # noqa: E402
from inputs import CONFIGS, VARIANT_CONFIGS, UNIT_EMBED, UNIT_FINAL_NORM, UNIT_LM_HEAD  # noqa: E402

ALL_CONFIGS = {**CONFIGS, **VARIANT_CONFIGS}

METRIC = "fine-tune tokens/sec at 1 GB300; % of step roofline (tensor peak vs host-link)"
UNIT = "tokens/s"


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["bf16_tflops"], d["bf16_tflops_sustained"], d["hbm_gbs"], "measured"
    return 1900.0, 1700.0, 6800.0, "fallback"


def layer_matmul_params(c):
    """P_m: the matmul parameters of one decoder layer."""
    q, kv = c.n_heads * c.head_dim, c.n_kv_heads * c.head_dim
    return c.hidden * q + 2 * c.hidden * kv + q * c.hidden + 3 * c.hidden * c.ffn


def attn_fwd_flops(c, batch=None):
    """Exact causal attention forward count (QK^T and PV over the causal
    half, diagonal included): 2 B Hq hd S (S + 1)."""
    B = c.batch if batch is None else batch
    return 2.0 * B * c.n_heads * c.head_dim * c.seq * (c.seq + 1)


def algorithmic_step_flops(c, n_micro=1):
    """F_step, the algorithmic work of one step: every decoder layer four
    times its forward (forward, recompute, backward = 2x forward) with the
    exact causal attention count, plus the fused head's three products
    (logits, dH, dW) over the valid rows: L 4 (2 P_m T + A) + 3 2 d V n_valid."""
    T = c.batch * c.seq
    n_valid = c.batch * (c.seq - 1)
    fwd = 2.0 * layer_matmul_params(c) * T + attn_fwd_flops(c)
    return n_micro * (c.n_layers * 4 * fwd + 3 * 2.0 * c.hidden * c.vocab * n_valid)


def step_flops(c, executed=True):
    """FLOPs the engine runs in one step: the recompute skips the down
    projection (its output is not needed) and the last layer is not
    recomputed; the head runs over all T rows (ignored rows included).
    executed=False gives algorithmic_step_flops."""
    if not executed:
        return algorithmic_step_flops(c)
    d, F, T = c.hidden, c.ffn, c.batch * c.seq
    q, kv = c.n_heads * c.head_dim, c.n_kv_heads * c.head_dim
    proj = {"qkv": 2 * T * d * (q + 2 * kv), "o": 2 * T * q * d, "gu": 2 * T * d * 2 * F, "down": 2 * T * F * d}
    attn = attn_fwd_flops(c)
    fwd = sum(proj.values()) + attn
    rec = fwd - proj["down"]
    bwd = 2 * sum(proj.values()) + 2.5 * attn
    layers = c.n_layers * fwd + (c.n_layers - 1) * rec + c.n_layers * bwd
    head = 3 * 2.0 * d * c.vocab * T
    return layers + head


def phase_bound_ms(c, peak_tflops, link, ring):
    """The phase-aware bound of a step: the sum over its phases of the slower
    of tensor work at peak and that phase's host-link copies, instead of the
    global max(F / peak, bytes / link).  Phases: each layer's forward (its
    weights' H2D of 2 P_l bytes hides under the previous layer's forward), the
    head (the LM head's H2D and its gradient's D2H), and each layer's
    recompute + backward (3x the forward; its gradients' D2H, plus the H2D of
    the layer R places earlier when that one is not resident, both ways at
    once)."""
    P = peak_tflops * 1e12
    P_l = layer_matmul_params(c) + 2 * c.hidden + (c.n_heads + 2 * c.n_kv_heads) * c.head_dim * bool(c.qkv_bias)
    lay = 2.0 * P_l
    T = c.batch * c.seq
    fwd = (2.0 * layer_matmul_params(c) * T + attn_fwd_flops(c)) / P
    head_fl = 3 * 2.0 * c.hidden * c.vocab * c.batch * (c.seq - 1) / P
    wlm = 2.0 * c.vocab * c.hidden
    bw = {k: v * 1e9 for k, v in link.items()}
    t = c.n_layers * max(fwd, lay / bw["h2d"])
    t += max(head_fl, wlm / bw["h2d"] + wlm / bw["d2h"])
    R = min(ring, c.n_layers)
    for l in range(c.n_layers - 1, -1, -1):
        link_t = (2 * lay / bw["bidir"]) if l - R >= 0 else lay / bw["d2h"]
        t += max(3 * fwd, link_t)
    return t * 1e3


def gemm_traffic_summary(path=None):
    """Per-launch DRAM traffic of the step's GEMMs from the committed ncu
    summary, if it was taken of the GEMM source as it stands (its SHA-256
    prefix is recorded beside the number); else None."""
    import hashlib
    import re
    path = path or os.path.join(ROOT, "profiles", "gemm_8b_step_traffic.md")
    src = os.path.join(ROOT, "offloaded_fine_tuning_gb300", "csrc", "gemm.cu")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    m = re.search(r"gemm_cu_sha256_16:\s*([0-9a-f]{16})", text)
    b = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    a = re.search(r"algorithmic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not (m and b) or m.group(1) != sha:
        return None
    return {"bytes": float(b.group(1)), "algorithmic": float(a.group(1)) if a else None,
            "source": os.path.relpath(path, ROOT)}


class ClockSampler:
    """nvidia-smi samples during the timed region (SM clock and throttle reasons)."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        self.index, self.rows, self.proc = index, [], None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")])

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = [r for r in self.rows if len(r) >= 9]
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        busy = [s for s in sm if mx and s > 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(busy) if busy else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


def job_throughput(tokens_per_step, steps, elapsed_ms):
    """Tokens/s of the whole job: every step's tokens over the timed region."""
    return tokens_per_step * steps / (elapsed_ms / 1e3)


def world_size(args) -> int:
    return max(int(os.environ.get("WORLD_SIZE", "1")), args.gpus)


def refuse_multi_gpu(args) -> bool:
    """True (after rank 0 printed why) when the launch asks for more than one
    GPU: the library is single-GPU by design (its GEMMs multicast weight
    tiles between the two CTAs of a cluster, inside one GPU's memory)."""
    n = world_size(args)
    if n <= 1:
        return False
    if int(os.environ.get("RANK", "0")) == 0:
        print(json.dumps({"metric": METRIC, "unit": UNIT, "n_gpus": n, "impl": args.impl,
                          "unavailable": "single-GPU library: the layer-sliding step runs on one "
                                         "GPU (GEMM clusters multicast tiles within that GPU's "
                                         "memory; no cross-GPU path is built)"}), flush=True)
    return True


def link_probe(torch, nbytes=1 << 30):
    """Pinned host<->device GB/s: H2D, D2H and both directions at once."""
    h1 = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    h2 = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d1 = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    d2 = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    out = {}
    for name, fn in (("h2d", lambda: d1.copy_(h1, non_blocking=True)),
                     ("d2h", lambda: h2.copy_(d2, non_blocking=True))):
        fn(); torch.cuda.synchronize()
        t = time.perf_counter()
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        out[name] = 3 * nbytes / (time.perf_counter() - t) / 1e9
    torch.cuda.synchronize()
    t = time.perf_counter()
    for _ in range(3):
        with torch.cuda.stream(s1):
            d1.copy_(h1, non_blocking=True)
        with torch.cuda.stream(s2):
            h2.copy_(d2, non_blocking=True)
    torch.cuda.synchronize()
    out["bidir"] = 6 * nbytes / (time.perf_counter() - t) / 1e9
    del h1, h2, d1, d2
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------------ oracle sample (CPU)
def oracle_sample(c, reps=1):
    """Time the CPU oracle (float32, as it stands) on a bounded sample of the
    workload: one sequence through one full-shape decoder layer forward and
    backward plus the LM head and loss on its rows.  Returns (tokens/s of the
    whole step extrapolated to n_layers, seconds, description)."""
    import oracle
    from oracle import llama_step as ls
    cs = c.with_(n_layers=1, batch=1)
    S, d = cs.seq, cs.hidden
    lay = {k: oracle.bf16_round(v) for k, v in inputs.split_layer(cs, inputs.layer_master(cs, 0)).items()}
    Wlm = oracle.bf16_round(inputs.normal(1234, 2, c.vocab * d, 0.0, 0.02)).reshape(c.vocab, d)
    gf = np.ones(d, np.float32)
    tok, lab = inputs.tokens_and_labels(cs)
    x = inputs.normal(1234, 3, S * d, 0.0, 0.02).reshape(1, S, d)
    cos, sin = ls.rope_tables(S, c.head_dim, c.rope_base, np.float32)
    t_layer = t_head = 0.0
    for _ in range(reps):
        t0 = time.perf_counter()
        y, cache = ls.layer_fwd(x, lay, cs, cos, sin)
        t1 = time.perf_counter()
        hf, cf = ls.rmsnorm_fwd(y.reshape(S, d), gf, cs.rms_eps)
        z = hf @ Wlm.T
        _, dz, _ = ls.cross_entropy_fwd_bwd(z, lab.reshape(-1))
        _ = dz.T @ hf
        dh, _ = ls.rmsnorm_bwd(dz @ Wlm, gf, cf)
        t2 = time.perf_counter()
        ls.layer_bwd(dh.astype(np.float32), lay, cache, cs, cos, sin)
        t3 = time.perf_counter()
        t_layer += (t1 - t0) + (t3 - t2)
        t_head += t2 - t1
    t_layer /= reps
    t_head /= reps
    # the full step also recomputes each layer's forward once: count it
    t_fwd = t_layer / 3.0
    t_step = c.batch * (c.n_layers * (t_layer + t_fwd) + t_head)
    desc = (f"1 sequence x {S} tokens through one {c.name} decoder layer fwd+bwd "
            f"({t_layer:.1f}s) and the LM head + loss ({t_head:.1f}s), float32 numpy; "
            f"extrapolated to {c.n_layers} layers (+recompute) x batch {c.batch}")
    return c.batch * S / t_step, t_layer + t_head, desc


def oracle_full_step(c):
    """Time one whole CPU oracle step (float32) of a small workload as it is:
    returns (tokens/s, seconds, description)."""
    import oracle
    d, V = c.hidden, c.vocab
    layers = [{k: oracle.bf16_round(v) for k, v in inputs.split_layer(c, inputs.layer_master(c, l)).items()}
              for l in range(c.n_layers)]
    r = lambda u: oracle.bf16_round(inputs.unit_master(c, u))
    w = oracle.ModelWeights(layers=layers, embed=r(UNIT_EMBED).reshape(V, d), final_norm=r(UNIT_FINAL_NORM),
                            lm_head=r(UNIT_LM_HEAD).reshape(V, d))
    tok, lab = inputs.tokens_and_labels(c)
    t0 = time.perf_counter()
    oracle.step(w, tok, lab, c, dtype=np.float32)
    secs = time.perf_counter() - t0
    return c.batch * c.seq / secs, secs, f"the whole {c.name} step ({c.batch} x {c.seq} tokens), float32 numpy"


def oracle_lce_sample(c, rows=1024):
    """Time the CPU oracle's unfused LM head + cross-entropy forward and
    backward on a block of rows of the large-vocabulary workload, float32:
    returns (rows/s of the whole workload, seconds, description)."""
    import oracle
    h, w, lab = inputs.lce_inputs(c)
    W = oracle.bf16_round(w)
    hb = oracle.bf16_round(h[:rows])
    t0 = time.perf_counter()
    _, dz, _ = oracle.cross_entropy_fwd_bwd(hb @ W.T, lab[:rows])
    _ = dz @ W
    _ = dz.T @ hb
    secs = time.perf_counter() - t0
    n = c.batch * c.seq
    return rows / secs, secs, (f"{rows} of {n} rows of {c.name}: logits, loss, dH and dW "
                               f"(float32 numpy), rows/s")


def oracle_timings():
    """The CPU oracle, as it stands, on a bounded sample of every other
    workload (the tiny one whole; one sequence through one layer plus the
    head, extrapolated, for the decoder stacks; a block of rows for the
    large-vocabulary head)."""
    from inputs import LCE_STRESS
    out = {}
    for name in ("tiny", "1.3b", "123b-slice"):
        c = CONFIGS[name]
        v, secs, desc = oracle_full_step(c) if name == "tiny" else oracle_sample(c)
        out[c.name] = {"value": v, "unit": UNIT, "seconds": secs, "sample": desc}
    v, secs, desc = oracle_lce_sample(LCE_STRESS)
    out[LCE_STRESS.name] = {"value": v, "unit": UNIT, "seconds": secs, "sample": desc}
    return out


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def run_reference(args, c):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    for _ in range(args.warmup):
        oracle_sample(c)
    vals, secs = [], 0.0
    for _ in range(args.steps):
        v, s, desc = oracle_sample(c)
        vals.append(v)
        secs += s
    value = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": c.batch * c.seq / value * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": c.name, "global_batch": c.batch, "seq_len": c.seq,
                       "parallelism": "cpu oracle"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ our arm
def load_model(sf, c, ring, async_update, offload_activations=0, bf16_adam_state=0):
    cfg = sf.make_config(c, ring_slots=ring, retain_grads=0, async_update=async_update,
                         offload_activations=offload_activations, bf16_adam_state=bf16_adam_state)
    m = sf.Model(cfg)
    for l in range(c.n_layers):
        m.load(l, inputs.layer_master(c, l))
    for u in (UNIT_EMBED, UNIT_FINAL_NORM, UNIT_LM_HEAD):
        if inputs.unit_numel(c, u):  # no LM-head unit when it is tied
            m.load(u, inputs.unit_master(c, u))
    return m


def host_adam_bytes(c, micro=1, bf16_state=False):
    """Host memory traffic of one step's updates.  Layers, final norm and an
    untied LM head: 28 B per parameter (bf16 gradient in, fp32 master, m, v
    read and written, bf16 pack out).  Embedding: 24 B (fp32 gradient, state)
    plus, when it is the tied head, 6 B to fold the head's bf16 gradient into
    it.  Each extra micro-batch adds 12 B per packed parameter (bf16 gradient
    in, fp32 sum read and written, bf16 weights back)."""
    P_l = inputs.unit_numel(c, 0)
    packed = c.n_layers * P_l + c.hidden + inputs.unit_numel(c, UNIT_LM_HEAD)
    emb = c.vocab * c.hidden
    s = 8.0 if bf16_state else 0.0  # bf16 moments: 2 + 2 bytes read and written instead of 4 + 4
    b = (28.0 - s) * packed + (24.0 - s) * emb + (6.0 * emb if c.tie_embeddings else 0.0)
    return b + (micro - 1) * 12.0 * (packed + (emb if c.tie_embeddings else 0))


def run_ours(args, c):
    import torch
    import offloaded_fine_tuning_gb300 as sf
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    sf.lib(build_if_needed=True)
    bf16_peak, bf16_sust, hbm, peak_src = peaks()
    link = link_probe(torch)
    host_gbs = sf.probe_host_bandwidth(0, 8 << 30)

    m = load_model(sf, c, args.ring or c.ring_slots, 0 if args.sync_updates else 1,
                   1 if args.offload_activations else 0, 1 if args.bf16_adam_state else 0)
    adam = sf.Adam(lr=1e-5, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0)
    # a fresh batch each step; with --micro N
    # a step is N micro-batches of the workload's batch, summed before the update
    n_micro = max(1, args.micro)
    n_batches = args.warmup + 2 * args.steps

    def make_batch(i):
        parts = [inputs.tokens_and_labels(c, seed=inputs.SEED_TOKENS + n_micro * i + j)
                 for j in range(n_micro)]
        if n_micro == 1:
            return parts[0]
        return np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts])

    batches = [make_batch(i) for i in range(n_batches)]
    T = n_micro * c.batch * c.seq

    def train(tok, lab):
        return m.train_step(tok, lab, adam) if n_micro == 1 else m.train_step_accum(tok, lab, adam)

    for i in range(args.warmup):
        assert train(*batches[i]) == sf.SF_OK, m.error()

    m.sync()  # no warm-up update runs into the timed region
    m.trace()  # start the host timeline at the timed region
    # ---- device-clock region (CUDA events, host Adam included): K steps
    m.set_timing(True)
    clocks = ClockSampler(local)
    clocks.start()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    stats = []
    for i in range(args.steps):
        st = train(*batches[args.warmup + i])
        assert st == sf.SF_OK, m.error()
        stats.append(m.stats())
    m.sync()  # the last step's host updates belong to the timed work
    e1.record()
    timeline = m.trace()
    torch.cuda.synchronize()
    dev_ms = e0.elapsed_time(e1)
    clk = clocks.stop()
    m.set_timing(False)

    # ---- end to end through the public call: stage the batch from pinned host
    # memory each step, run the step, read the loss back
    shape = (c.batch, c.seq) if n_micro == 1 else (n_micro, c.batch, c.seq)
    pin_tok = torch.empty(shape, dtype=torch.int32, pin_memory=True)
    pin_lab = torch.empty(shape, dtype=torch.int32, pin_memory=True)
    t0 = time.perf_counter()
    losses = []
    for i in range(args.steps):
        tok, lab = batches[args.warmup + args.steps + i]
        pin_tok.numpy()[...] = tok
        pin_lab.numpy()[...] = lab
        assert train(pin_tok.numpy(), pin_lab.numpy()) == sf.SF_OK, m.error()
        losses.append(m.loss())
    m.sync()
    e2e_s = time.perf_counter() - t0

    # the GPU path alone: two steps without the optimizer (no host Adam), synchronous
    gpu_path_ms, gp_stats = None, []
    if not args.no_gpu_path:
        m.sync()
        torch.cuda.synchronize()
        g0 = time.perf_counter()
        for i in range(2):
            tok, lab = batches[args.warmup + i]
            st = m.train_step(tok, lab) if n_micro == 1 else m.train_step_accum(tok, lab)
            assert st == sf.SF_OK, m.error()
        gpu_path_ms = (time.perf_counter() - g0) * 1e3 / 2
        # the same steps with the engine's event timeline: the compute stream's
        # waits are then waits for copies alone (no host update to wait for)
        m.set_timing(True)
        for i in range(2):
            tok, lab = batches[args.warmup + i]
            st = m.train_step(tok, lab) if n_micro == 1 else m.train_step_accum(tok, lab)
            assert st == sf.SF_OK, m.error()
            gp_stats.append(m.stats())
        m.set_timing(False)

    e2e_ms = e2e_s * 1e3
    ms_step = dev_ms / args.steps
    value = job_throughput(T, args.steps, dev_ms)
    e2e = job_throughput(T, args.steps, e2e_ms)

    gemm_ms = sum(s["gemm_ms"] for s in stats)
    gemm_fl = sum(s["gemm_flops"] for s in stats)
    gemm_n = sum(s["gemm_launches"] for s in stats)
    attn_ms = sum(s["attn_ms"] for s in stats)
    attn_fl = sum(s["attn_flops"] for s in stats)
    # the engine's counters cover the last micro-batch of a step
    h2d = n_micro * statistics.mean(s["h2d_bytes"] for s in stats)
    d2h = n_micro * statistics.mean(s["d2h_bytes"] for s in stats)
    gpu_step = n_micro * statistics.mean(s["step_ms"] for s in stats)
    achieved = gemm_fl / (gemm_ms / 1e3) / 1e12 if gemm_ms > 0 else None
    F_exec = n_micro * step_flops(c, executed=True)
    F_step = algorithmic_step_flops(c, n_micro)
    t_tensor = F_step / (bf16_sust * 1e12)
    t_link = (h2d + d2h) / (link["bidir"] * 1e9)
    t_roof = max(t_tensor, t_link)
    t_phase = n_micro * phase_bound_ms(c, bf16_sust, link, args.ring or c.ring_slots)
    exposed = n_micro * statistics.mean(s["exposed_ms"] for s in stats)
    traffic = gemm_traffic_summary()
    n_launch = n_micro * gemm_n / args.steps
    # host memory: the Adam update of every unit (28 B per layer / LM-head
    # parameter: bf16 grad in, fp32 master, m, v read and written, bf16 out;
    # 24 B per embedding parameter, whose gradient is fp32) plus the DMA copies
    adam_bytes = host_adam_bytes(c, n_micro, args.bf16_adam_state)
    host_bytes = adam_bytes + h2d + d2h
    t_host = host_bytes / (host_gbs * 1e9)
    if args.trace:
        with open(args.trace, "w") as f:
            json.dump(timeline, f)
    cpu = None
    if not args.no_cpu_baseline:
        v, secs, desc = oracle_sample(c)
        cpu = {"value": v, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle", "sample": desc,
               "other_workloads": oracle_timings()}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": c.name, "global_batch": n_micro * c.batch, "seq_len": c.seq,
                   "micro_batches": n_micro,
                   "layers": c.n_layers, "ring_slots": args.ring or c.ring_slots,
                   "parallelism": "single-gpu layer sliding",
                   "host_updates": "synchronous" if args.sync_updates else "overlap next step",
                   "activations": "sliding (host)" if args.offload_activations else "resident",
                   "adam_state": "bf16, stochastic rounding" if args.bf16_adam_state else "fp32",
                   "l2": "inputs larger than L2 (each step streams every layer's weights and gradients)"},
        "e2e": {"value": e2e, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_ms / args.steps},
        "gpu_launches": int(n_micro * sum(s["kernel_launches"] for s in stats)),
        "roofline": {"kernel": "gemm_tcgen05", "bound": "tensor", "achieved": achieved,
                     "peak": bf16_sust, "unit": "TFLOP/s",
                     "frac": achieved / bf16_sust if achieved else None,
                     "traffic": traffic["bytes"] if traffic else None,
                     "traffic_algorithmic": traffic["algorithmic"] if traffic else None,
                     "traffic_source": traffic["source"] if traffic else
                     "no ncu capture of the current GEMM source",
                     "flops_per_launch": gemm_fl / max(1, gemm_n),
                     "peak_source": f"{peak_src} bf16 sustained (cuBLAS, long loop)",
                     "launches_per_step": n_launch,
                     "gemm_ms_per_step": n_micro * gemm_ms / args.steps},
        "step_roofline": {"flops": F_step, "flops_executed": F_exec,
                          "t_tensor_ms": t_tensor * 1e3, "h2d_bytes": h2d,
                          "d2h_bytes": d2h, "link_gbs": link, "t_link_ms": t_link * 1e3,
                          "t_roof_ms": t_roof * 1e3, "frac": t_roof * 1e3 / ms_step,
                          "phase_bound_ms": t_phase, "phase_frac": t_phase / ms_step,
                          "exposed_copy_ms": n_micro * statistics.mean(x["exposed_ms"] for x in gp_stats)
                          if gp_stats else None,
                          "exposed_copy_what": "compute-stream time not covered by layer and head "
                                               "compute in the steps without the optimizer (waits for "
                                               "weight, checkpoint and batch copies)",
                          "compute_stream_wait_ms": exposed,
                          "compute_stream_wait_what": "the same in the timed steps, where a layer's "
                                                      "weight copy also waits for its host update",
                          "compute_stream_ms": n_micro * statistics.mean(s["compute_ms"] for s in stats),
                          "head_ms": n_micro * statistics.mean(s["head_ms"] for s in stats),
                          "host_memory": {"bytes": host_bytes, "adam_bytes": adam_bytes,
                                          "probe_gbs": host_gbs, "t_ms": t_host * 1e3,
                                          "frac": t_host * 1e3 / ms_step},
                          "gpu_busy_ms": gpu_step,
                          "attn_tflops": attn_fl / (attn_ms / 1e3) / 1e12 if attn_ms > 0 else None,
                          "host_adam_ms": statistics.mean(s["host_adam_ms"] for s in stats),
                          "host_tail_ms": statistics.mean(s["host_wait_ms"] for s in stats)},
        "gpu_path": None if gpu_path_ms is None else {
            "ms_per_step": gpu_path_ms, "tokens_per_s": T / (gpu_path_ms / 1e3),
            "what": "same step without the optimizer update (no host Adam), host wall clock"},
        "clocks": clk,
        "loss": losses[-1],
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    m.close()


def run_lce(args):
    """The large-vocabulary LM head + cross-entropy workload (4 x 4096 rows of
    hidden 3584, vocabulary 152064, 10% of labels ignored): value = rows/s of
    the fused chunked forward + backward on device-resident inputs (CUDA
    events; W alone is 1.09 GB, larger than L2); e2e = the same through
    sf_lce_step on host buffers (its H2D of h, W, labels and D2H of loss, dH,
    dW inside the timed region)."""
    import torch
    import offloaded_fine_tuning_gb300 as sf
    from inputs import LCE_STRESS as c
    sf.lib(build_if_needed=True)
    bf16_peak, bf16_sust, hbm, peak_src = peaks()
    h, w, lab = inputs.lce_inputs(c)
    n, d, V = h.shape[0], c.hidden, c.vocab
    bits = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16)
    hb, wb = bits(h), bits(w)
    H, W, Y = hb.cuda(), wb.cuda(), torch.from_numpy(lab.astype(np.int32)).cuda()
    n_valid = int(np.sum(lab != sf.IGNORE_INDEX))
    cap = max(128, ((2 << 30) // (6 * V)) // 128 * 128)  # as the library's automatic chunk
    chunks = -(-n // cap)
    chunk = min(n, (-(-n // chunks) + 127) // 128 * 128)
    ws = torch.empty(sf.lce_workspace_bytes(n, V, chunk), dtype=torch.uint8, device="cuda")
    loss = torch.empty(1, device="cuda")
    dh = torch.empty((n, d), device="cuda")
    dw = torch.empty((V, d), device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    run = lambda: sf.op_lce(H.data_ptr(), W.data_ptr(), Y.data_ptr(), n, d, V, n_valid, chunk,
                            ws.data_ptr(), loss.data_ptr(), dh.data_ptr(), dw.data_ptr(), st)
    for _ in range(args.warmup):
        assert run() == 0
    torch.cuda.synchronize()
    clocks = ClockSampler(int(os.environ.get("LOCAL_RANK", "0")))
    clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        run()
    e1.record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    assert sf.device_error() == 0
    ms = e0.elapsed_time(e1) / args.steps
    launches_per_step = sf.lce_launches()
    # end to end through the public call on host buffers (bf16 bits), in
    # page-locked memory as a training loop would keep them
    hbits = hb.view(torch.int16).pin_memory().numpy().view(np.uint16)
    wbits = wb.view(torch.int16).pin_memory().numpy().view(np.uint16)
    labp = torch.from_numpy(lab.astype(np.int32)).pin_memory().numpy()
    dh_host = torch.empty((n, d), dtype=torch.int16).pin_memory().numpy().view(np.uint16)
    dw_host = torch.empty((V, d), dtype=torch.float32).pin_memory().numpy()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        l_host, _, _ = sf.lce_step(hbits, wbits, labp, dh_out=dh_host, dw_out=dw_host)
    e2e_s = (time.perf_counter() - t0) / args.steps
    flops = 3 * 2.0 * n * V * d
    tf = flops / (ms / 1e3) / 1e12
    cpu = None
    if not args.no_cpu_baseline:
        v, secs, desc = oracle_lce_sample(c)
        cpu = {"value": v, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle", "sample": desc}
    line = {
        "metric": METRIC, "value": n / (ms / 1e3), "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": c.name, "global_batch": c.batch, "seq_len": c.seq, "hidden": d,
                   "vocab": V, "ignored": c.ignore_frac, "chunk_rows": chunk,
                   "parallelism": "single-gpu", "l2": "inputs larger than L2 (W_lm 1.09 GB)",
                   "what": "fused chunked LM head + cross-entropy forward and backward (tokens = rows)"},
        "e2e": {"value": n / e2e_s, "unit": UNIT, "ms_per_step": e2e_s * 1e3,
                "h2d_bytes_per_step": n * d * 2 + V * d * 2 + n * 4,
                "d2h_bytes_per_step": 4 + n * d * 2 + V * d * 4},
        "gpu_launches": args.steps * launches_per_step,
        "roofline": {"kernel": "fused LM head (3 GEMMs per chunk + row softmax)", "bound": "tensor",
                     "achieved": tf, "peak": bf16_peak, "unit": "TFLOP/s", "frac": tf / bf16_peak,
                     "traffic": None, "flops_per_step": flops,
                     "peak_source": f"{peak_src} bf16 burst (one op timed alone)"},
        "clocks": clk, "loss": float(loss.item()), "loss_e2e": l_host, "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


def run_reference_lce(args):
    """--impl reference on the large-vocabulary workload: the CPU oracle on a
    block of rows per step, as it stands."""
    from inputs import LCE_STRESS as c
    if int(os.environ.get("RANK", "0")) != 0:
        return
    for _ in range(args.warmup):
        oracle_lce_sample(c)
    vals = []
    for _ in range(args.steps):
        v, secs, desc = oracle_lce_sample(c)
        vals.append(v)
    value = statistics.median(vals)
    n = c.batch * c.seq
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": n / value * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": {"workload": c.name, "global_batch": c.batch, "seq_len": c.seq,
                                        "parallelism": "cpu oracle"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
        flush=True)


def run_op(args, c):
    """Time one kernel at the workload's shapes on device-resident data (CUDA
    events on the launching stream, inputs larger than L2).  Prints one JSON line."""
    import torch
    import offloaded_fine_tuning_gb300 as sf
    sf.lib(build_if_needed=True)
    torch.manual_seed(0)
    st = torch.cuda.current_stream().cuda_stream
    B, S, Hq, Hkv, hd = c.batch, c.seq, c.n_heads, c.n_kv_heads, c.head_dim
    T = B * S
    W = (Hq + 2 * Hkv) * hd
    attn_fwd_flops = 2.0 * B * Hq * hd * S * (S + 1)
    bf16_peak, bf16_sust, hbm, src = peaks()
    if args.op in ("rmsnorm_fwd", "rmsnorm_bwd", "rope", "swiglu_fwd", "swiglu_bwd"):
        return run_op_hbm(args, c, sf, torch, st, hbm, src)
    if args.op.startswith("attn"):
        qkv = torch.randn(T, W, device="cuda").to(torch.bfloat16)
        o = torch.empty(T, Hq * hd, device="cuda", dtype=torch.bfloat16)
        lse = torch.empty(B, Hq, S, device="cuda")
        dout = torch.randn(T, Hq * hd, device="cuda").to(torch.bfloat16)
        dqkv = torch.empty_like(qkv)
        delta = torch.empty(B, Hq, S, device="cuda")
        dqa = torch.empty(T, Hq * hd, device="cuda")
        fwd = lambda: sf.op_attn_fwd(qkv.data_ptr(), o.data_ptr(), lse.data_ptr(), B, S, Hq, Hkv, hd, st)
        bwd = lambda: sf.op_attn_bwd(qkv.data_ptr(), o.data_ptr(), dout.data_ptr(), lse.data_ptr(),
                                     delta.data_ptr(), dqa.data_ptr(), dqkv.data_ptr(), B, S, Hq, Hkv, hd, 0, st)
        assert fwd() == 0
        run, flops = (fwd, attn_fwd_flops) if args.op == "attn_fwd" else (bwd, 2.5 * attn_fwd_flops)
        shape = {"B": B, "S": S, "Hq": Hq, "Hkv": Hkv, "hd": hd}
    else:
        M, N, K = (int(x) for x in args.shape.split(","))
        layout = {"nt": sf.NT, "nn": sf.NN, "tn": sf.TN}[args.layout]
        a_shape = (K, M) if layout == sf.TN else (M, K)
        b_shape = (N, K) if layout == sf.NT else (K, N)
        A = torch.randn(*a_shape, device="cuda").to(torch.bfloat16)
        Bm = torch.randn(*b_shape, device="cuda").to(torch.bfloat16)
        C = torch.empty(M, N, device="cuda", dtype=torch.bfloat16)
        run = lambda: sf.op_gemm(layout, sf.EPI_BF16, M, N, K, A.data_ptr(), a_shape[1], Bm.data_ptr(),
                                 b_shape[1], C.data_ptr(), N, 0, 0, 1.0, st)
        flops = 2.0 * M * N * K
        shape = {"M": M, "N": N, "K": K, "layout": args.layout}
    for _ in range(args.warmup):
        assert run() == 0
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        run()
    e1.record()
    torch.cuda.synchronize()
    assert sf.device_error() == 0
    ms = e0.elapsed_time(e1) / args.steps
    tf = flops / (ms / 1e3) / 1e12
    print(json.dumps({"op": args.op, "workload": c.name, "shape": shape, "ms": ms, "tflops": tf,
                      "peak": bf16_peak, "frac": tf / bf16_peak,
                      "peak_source": f"{src} bf16 burst (kernel timed alone)"}), flush=True)


def run_op_hbm(args, c, sf, torch, st, hbm, src):
    """The memory-bound kernels of a decoder layer at the workload's shapes:
    time per launch and algorithmic bytes (each tensor read or written once)
    against the measured HBM copy bandwidth."""
    T, d, F = c.batch * c.seq, c.hidden, c.ffn
    q, kv = c.n_heads * c.head_dim, c.n_kv_heads * c.head_dim
    bf = torch.bfloat16
    dev = "cuda"
    if args.op == "rmsnorm_fwd":
        x = torch.randn(T, d, device=dev)
        g = torch.ones(d, device=dev, dtype=bf)
        y = torch.empty(T, d, device=dev, dtype=bf)
        rstd = torch.empty(T, device=dev)
        run = lambda: sf.op_rmsnorm_fwd(x.data_ptr(), g.data_ptr(), y.data_ptr(), rstd.data_ptr(), T, d, c.rms_eps, st)
        nbytes = T * d * (4 + 2) + T * 4 + d * 2
        shape = {"rows": T, "d": d, "bytes": "x fp32 in, y bf16 + rstd out"}
    elif args.op == "rmsnorm_bwd":
        x, dy, dres = (torch.randn(T, d, device=dev) for _ in range(3))
        g = torch.ones(d, device=dev, dtype=bf)
        rstd = torch.ones(T, device=dev)
        dx = torch.empty(T, d, device=dev)
        dxb = torch.empty(T, d, device=dev, dtype=bf)
        dg = torch.empty(d, device=dev, dtype=bf)
        scr = torch.empty(sf.rmsnorm_bwd_scratch(T, d), device=dev)
        run = lambda: sf.op_rmsnorm_bwd(x.data_ptr(), g.data_ptr(), rstd.data_ptr(), dy.data_ptr(), dres.data_ptr(),
                                        dx.data_ptr(), dxb.data_ptr(), dg.data_ptr(), scr.data_ptr(), T, d, st)
        nbytes = T * d * (4 + 4 + 4 + 4 + 2) + T * 4 + d * 2
        shape = {"rows": T, "d": d, "bytes": "x, dy, residual grad fp32 in; dx fp32 + bf16 out"}
    elif args.op == "rope":
        W = q + 2 * kv
        x = torch.randn(T, W, device=dev).to(bf)
        tab = torch.from_numpy(sf.rope_table(c.seq, c.head_dim, c.rope_base)).to(dev)
        run = lambda: sf.op_rope(x.data_ptr(), W, T, c.seq, c.n_heads + c.n_kv_heads, c.head_dim,
                                 tab.data_ptr(), 0, st)
        nbytes = T * (q + kv) * 2 * 2
        shape = {"tokens": T, "heads": c.n_heads + c.n_kv_heads, "hd": c.head_dim, "bytes": "Q, K bf16 read and written in place"}
    elif args.op == "swiglu_fwd":
        ab = torch.randn(T, 2 * F, device=dev).to(bf)
        m = torch.empty(T, F, device=dev, dtype=bf)
        run = lambda: sf.op_swiglu_fwd(ab.data_ptr(), m.data_ptr(), T, F, st)
        nbytes = T * F * (4 + 2)
        shape = {"rows": T, "ffn": F, "bytes": "[a|b] bf16 in, m bf16 out"}
    else:
        ab = torch.randn(T, 2 * F, device=dev).to(bf)
        dm = torch.randn(T, F, device=dev).to(bf)
        dab = torch.empty(T, 2 * F, device=dev, dtype=bf)
        run = lambda: sf.op_swiglu_bwd(dm.data_ptr(), ab.data_ptr(), dab.data_ptr(), T, F, st)
        nbytes = T * F * (2 + 4 + 4)
        shape = {"rows": T, "ffn": F, "bytes": "dm, [a|b] bf16 in, [da|db] bf16 out"}
    for _ in range(args.warmup):
        assert run() == 0
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        run()
    e1.record()
    torch.cuda.synchronize()
    assert sf.device_error() == 0
    ms = e0.elapsed_time(e1) / args.steps
    gbs = nbytes / (ms / 1e3) / 1e9
    print(json.dumps({"op": args.op, "workload": c.name, "shape": shape, "ms": ms,
                      "algorithmic_bytes": nbytes, "gbs": gbs, "peak": hbm, "frac": gbs / hbm,
                      "peak_source": f"{src} HBM copy bandwidth"}), flush=True)


def run_sweep(args, c):
    """The overlap condition of the layer-sliding backward: per decoder layer,
    is the GPU backward (with its recompute) at least as long as copying the
    layer's gradients to the host plus the host Adam update?  Measured per
    batch size; the critical batch is the smallest one where it holds."""
    import torch
    import offloaded_fine_tuning_gb300 as sf
    sf.lib(build_if_needed=True)
    batches = [int(x) for x in args.sweep_batch.split(",")]
    cfg = sf.make_config(c, max_batch=max(batches), ring_slots=args.ring or c.ring_slots,
                         retain_grads=0, async_update=0)
    m = sf.Model(cfg)
    for l in range(c.n_layers):
        m.load(l, inputs.layer_master(c, l))
    for u in (UNIT_EMBED, UNIT_FINAL_NORM, UNIT_LM_HEAD):
        m.load(u, inputs.unit_master(c, u))
    adam = sf.Adam(lr=1e-5, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0)
    rows = []
    for B in batches:
        cb = c.with_(batch=B)
        tok, lab = inputs.tokens_and_labels(cb, seed=inputs.SEED_TOKENS + B)
        m.set_timing(False)
        for _ in range(args.warmup):
            assert m.train_step(tok, lab, adam) == sf.SF_OK, m.error()
        m.set_timing(True)
        st = []
        t0 = time.perf_counter()
        for _ in range(args.steps):
            assert m.train_step(tok, lab, adam) == sf.SF_OK, m.error()
            st.append(m.stats())
        wall = (time.perf_counter() - t0) / args.steps
        avg = {k: statistics.mean(x[k] for x in st) for k in
               ("fwd_layer_ms", "bwd_layer_ms", "d2h_layer_ms", "update_layer_ms")}
        need = avg["d2h_layer_ms"] + avg["update_layer_ms"]
        rows.append({"batch": B, "tokens": B * c.seq, **{k: round(v, 3) for k, v in avg.items()},
                     "d2h_plus_update_ms": round(need, 3), "overlapped": avg["bwd_layer_ms"] >= need,
                     "step_ms": round(wall * 1e3, 1), "tokens_per_s": round(B * c.seq / wall, 1)})
        print(json.dumps(rows[-1]), flush=True)
    crit = None
    for a, b in zip(rows, rows[1:]):
        fa = a["bwd_layer_ms"] - a["d2h_plus_update_ms"]
        fb = b["bwd_layer_ms"] - b["d2h_plus_update_ms"]
        if fa < 0 <= fb:
            crit = a["batch"] + (b["batch"] - a["batch"]) * (-fa) / (fb - fa)
    if crit is None and rows and rows[0]["overlapped"]:
        crit = rows[0]["batch"]
    if crit is None and len(rows) >= 2:  # extrapolate the (linear in batch) backward time
        a, b = rows[-2], rows[-1]
        slope = (b["bwd_layer_ms"] - a["bwd_layer_ms"]) / (b["batch"] - a["batch"])
        if slope > 0:
            crit = b["batch"] + (b["d2h_plus_update_ms"] - b["bwd_layer_ms"]) / slope
    print(json.dumps({"sweep": "critical batch", "workload": c.name, "seq_len": c.seq,
                      "critical_batch": crit, "condition": "T_bwd >= T_grad_d2h + T_update"}), flush=True)
    m.close()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", default="8b", choices=sorted(ALL_CONFIGS) + ["lce-stress"])
    ap.add_argument("--micro", type=int, default=1,
                    help="gradient accumulation: micro-batches (of the workload's batch) per step")
    ap.add_argument("--ring", type=int, default=0)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-gpu-path", action="store_true",
                    help="skip the two extra steps timed without the optimizer")
    ap.add_argument("--offload-activations", action="store_true",
                    help="sliding activations: layer checkpoints go to pinned host memory")
    ap.add_argument("--bf16-adam-state", action="store_true",
                    help="host Adam moments stored as bf16 with stochastic rounding")
    ap.add_argument("--sync-updates", action="store_true",
                    help="finish every host update before a step returns (no cross-step overlap)")
    ap.add_argument("--sweep-batch", default="",
                    help="comma-separated batch sizes: measure the backward overlap condition per layer")
    ap.add_argument("--trace", default="", help="write the host timeline of the timed steps (JSON)")
    ap.add_argument("--op", default="", choices=["", "attn_fwd", "attn_bwd", "gemm", "rmsnorm_fwd",
                                                 "rmsnorm_bwd", "rope", "swiglu_fwd", "swiglu_bwd"],
                    help="time one kernel instead of the training step")
    ap.add_argument("--shape", default="16384,6144,4096", help="M,N,K for --op gemm")
    ap.add_argument("--layout", default="nt", choices=["nt", "nn", "tn"])
    args = ap.parse_args()
    if args.config == "lce-stress":
        if args.impl == "reference":
            run_reference_lce(args)
        elif not refuse_multi_gpu(args):
            run_lce(args)
        return
    c = ALL_CONFIGS[args.config]
    if args.impl == "reference":
        # the CPU oracle: rank 0 alone runs it, on the host cores
        run_reference(args, c)
        return
    if refuse_multi_gpu(args):
        return
    if args.sweep_batch:
        run_sweep(args, c)
    elif args.op:
        run_op(args, c)
    else:
        run_ours(args, c)


if __name__ == "__main__":
    main()
