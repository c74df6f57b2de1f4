#!/usr/bin/env python
"""Decode-step benchmark: batch-1 greedy decode of the Llama-3.1-8B-shaped
Q8_0 model (32 layers, hidden 4096, 32/8 heads, head_dim 128, FFN 14336,
vocab 128256, seeded N(0, 0.02) weights) at KV context 2048 (``--ctx 8192``
for the long-context case), through the library's C ABI.

One "step" = one decode token: embedding, 32 layers (RMSNorm + QKV GEMV +
RoPE + KV append, split-K attention, O GEMV, gate/up GEMV, SwiGLU + down
GEMV), final norm, LM head GEMV and the greedy pick, all on the GPU.  The
weights (8.2 GB per token) are larger than L2, so no flush is needed between
steps.

Prints one JSON line.  ``--impl reference`` times the fp64 CPU oracle on the
same workload instead (one layer of the step per sample).  Under torchrun
each rank runs an independent replica (decode does not shard); rank 0
prints.  ``--workload`` selects the secondary measurements: prefill, fork
(shared-prefix fan-out), stream (70B with a device budget), skip (layer
skip), spec (self-speculative decoding), kquant (K-quant GEMV bandwidth),
batch (batched decode of 2/4/8 sequences).
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
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "decode tok/s, 8B-shape Q8_0 batch 1; achieved HBM GB/s as % of peak"

# ncu DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per launch
# of the dominant kernel, keyed by the sha256 prefix of the source file it
# was captured on (a changed kernel has no traffic figure until it is
# captured again); the captures are summarised under profiles/.
NCU_TRAFFIC = {
    # step.cu: 4-layer 8B Q8_0 model, ctx 2051, one step-kernel launch:
    # dram read 1,521,000,448 + write 5,145,344 B against 1,520,440,320
    # algorithmic bytes; the traffic grows with the layers, so a full launch
    # is scaled by the same ratio (the capture is summarised under profiles/)
    "37032cc45be1d22a": {"ratio": 1526145792 / 1520440320},
    # the same capture of the kernel with the 168-register cap: read
    # 1,521,014,784 + write 5,137,920 B against 1,520,440,320
    "47b42f33c1253915": {"ratio": 1526152704 / 1520440320},
}

KIND_NAMES = {1: "embed", 2: "gemv_qkv", 3: "attention", 4: "gemv_o", 5: "gemv_gate_up", 6: "gemv_down",
              7: "gemv_head", 8: "argmax", 9: "advance"}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=256)
    p.add_argument("--warmup", type=int, default=8)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--config", default="8b")
    p.add_argument("--ctx", type=int, default=2048)
    p.add_argument("--e2e-steps", type=int, default=32)
    p.add_argument("--profile-steps", type=int, default=4)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--profile-region", action="store_true",
                   help="bracket the timed decode region with cudaProfilerStart/Stop (for ncu --profile-from-start off)")
    p.add_argument("--layers", type=int, default=0,
                   help="keep only the first N layers (small cases for ncu captures; not a bench result)")
    p.add_argument("--skip-threshold", type=float, default=0.98,
                   help="layer skip workload: skip layers whose calibrated cosine exceeds this")
    p.add_argument("--kq-only", default="",
                   help="kquant workload: only this format and shape, e.g. q4_k:28672x8192 (small ncu captures)")
    p.add_argument("--draft-k", default="1,3,7",
                   help="speculative workload: draft lengths to time (comma-separated)")
    p.add_argument("--workload", choices=["decode", "prefill", "fork", "stream", "skip", "spec", "kquant", "batch",
                                          "h2d", "kmodel"],
                   default="decode",
                   help="decode (default, the headline line); the others are secondary measurements: "
                        "prefill (prompt of --ctx tokens), fork (shared prefix -> 8 branches), "
                        "stream (70B Q4_0 resident vs a 24 GB device budget), "
                        "skip (decode with the layers whose calibrated cosine exceeds --skip-threshold skipped), "
                        "spec (self-speculative greedy decoding vs plain greedy decoding; --config 70b: the 24 GB "
                        "budget with the resident layers as the draft), "
                        "kquant (Q4_K / Q6_K dequant-GEMV on the 70B projection shapes), "
                        "batch (batched decode of 2, 4 and 8 sequences at ctx --ctx: tok/s and per-kernel times)")
    return p.parse_args()


def peaks(key="hbm_gbs"):
    fallback = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d[key]), "measured"
    except Exception:
        return fallback[key], "fallback"


def load_config(name, layers):
    import dataclasses
    import synth
    cfg = synth.get_config(name)
    if layers:
        cfg = dataclasses.replace(cfg, n_layers=min(layers, cfg.n_layers))
    return cfg


def prefill_flops(cfg, T, pos0=0):
    """Algorithmic FLOPs of prefilling T tokens after pos0 cached ones: the
    projections, causal attention (scores and P V over keys 0..pos), and the
    LM head of the last token."""
    pairs = T * pos0 + T * (T + 1) // 2          # (query, key) pairs
    att = 2 * 2 * cfg.n_heads * cfg.head_dim * pairs
    return cfg.n_layers * (2 * cfg.layer_params() * T + att) + 2 * cfg.vocab * cfg.hidden


def _events(torch, stream, fn):
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    fn()
    e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / 1000.0


def max_over_ranks(ms, dist, device):
    """The slowest rank's time: every rank's replica must finish (barrier +
    max-over-ranks timing; decode runs as independent replicas, one per GPU,
    with no data-path collective)."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([float(ms)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world, steps_per_rank, ms):
    """Whole-job tokens/s: every rank decodes steps_per_rank tokens of its own
    replica in ms milliseconds (the max over ranks)."""
    return world * steps_per_rank / (ms / 1000.0)


def base_line(metric, value, unit, steps, warmup, ms, workload, extra):
    line = {"metric": metric, "value": round(value, 3), "unit": unit, "n_gpus": 1, "steps": steps,
            "warmup": warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int32+f32", "data": "synthetic", "config": {"workload": workload},
            "arith": "decode GEMVs: Q8_0/Q4_0 codes x int16-quantised activation slices, exact int32 dot products, "
                     "fp32 scaling and accumulation; tensor-core GEMMs: fp16 operand planes, fp32 accumulation; "
                     "fp16 KV cache"}
    line.update(extra)
    return line


def run_prefill(args):
    """Prompt processing: --steps prefills of --ctx tokens, each on a fresh sequence."""
    import torch
    import synth
    from decode_llama_step_gb300 import dls
    cfg = load_config(args.config, args.layers)
    w = synth.model_weights(cfg)
    stream = torch.cuda.Stream()
    m = dls.Model(cfg, w, max_seqs=2, max_ctx=args.ctx + 8, stream=stream)
    del w
    prompt = synth.prompt_tokens(cfg, args.ctx, seed=1)
    for _ in range(max(args.warmup, 1)):
        s = m.seq_create()
        m.prefill(s, prompt)
        m.seq_free(s)
    times = []
    with ClockSampler(0) as clk:
        for _ in range(args.steps):
            s = m.seq_create()
            times.append(_events(torch, stream, lambda: m.prefill(s, prompt)))
            m.seq_free(s)
    t = sum(times) / len(times)
    fl = prefill_flops(cfg, args.ctx)
    peak, src = peaks("bf16_tflops")
    peak_s, _ = peaks("bf16_tflops_sustained")
    m.close()
    extra = {"tensor": {"flops_per_prefill": fl, "achieved_tflops": round(fl / t / 1e12, 1),
                        "peak_tflops": peak, "frac": round(fl / t / 1e12 / peak, 4),
                        "frac_of_sustained": round(fl / t / 1e12 / peak_s, 4),
                        "peak_source": f"{src} bf16_tflops (fp16 operands run at the bf16 rate)"},
             "clocks": clk.summary()}
    if not args.no_cpu_baseline:
        tps, desc, cores = cpu_oracle_prefill_sample(cfg, args.ctx)
        extra["cpu_baseline"] = {"value": round(tps, 4), "unit": "tok/s", "cores": cores, "kind": "oracle",
                                 "sample": desc}
    return base_line(f"prefill tok/s, {cfg.name}-shape {'Q8_0' if cfg.wtype == 8 else 'Q4_0'}", args.ctx / t,
                     "tok/s", args.steps, args.warmup, 1000 * t,
                     f"{cfg.name} prefill of a {args.ctx}-token prompt (seeded ids) on an empty sequence", extra)


def run_fork(args):
    """Shared-prefix fork: one prefill of the prefix, a KV fork into 8
    branches and batch-8 greedy decode, against 8 independent prefills of
    the prefix followed by the same decode.  The headline value is the
    copying fork; the fork by shared pages is reported beside it."""
    import torch
    import synth
    from decode_llama_step_gb300 import dls
    cfg = load_config("fork8b", args.layers)
    P, B, D = cfg.workload["prefix"], cfg.workload["branches"], cfg.workload["decode"]
    w = synth.model_weights(cfg)
    stream = torch.cuda.Stream()
    m = dls.Model(cfg, w, max_seqs=B + 1, max_ctx=P + D + 8, max_batch=B, page_tokens=64, stream=stream)
    del w
    prefix = synth.prompt_tokens(cfg, P, seed=1)
    start = [100 + b for b in range(B)]
    s = m.seq_create()
    m.prefill(s, prefix[:256])
    m.generate([s], [1], 2)
    m.seq_free(s)
    with ClockSampler(0) as clk:
        src = m.seq_create()
        t_pre = _events(torch, stream, lambda: m.prefill(src, prefix))
        dsts = [m.seq_create() for _ in range(B)]
        t_fork = _events(torch, stream, lambda: m.kv_fork(src, dsts))
        m.generate(dsts, start, 2)  # capture the batch-8 graph outside the timing
        for d in dsts:
            m.seq_free(d)
        dsts = [m.seq_create() for _ in range(B)]
        m.kv_fork(src, dsts)
        t_dec = _events(torch, stream, lambda: m.generate(dsts, start, D))
        # per-kind device time of one batched step (kernels timed one by one)
        kms, kk = m.profile_batch(dsts, start, [m.seq_length(d) for d in dsts])
        per_kind = {}
        for d_ms, k in zip(kms, kk):
            e = per_kind.setdefault(KIND_NAMES.get(int(k), str(int(k))), {"launches_per_step": 0, "ms_per_step": 0.0})
            e["launches_per_step"] += 1
            e["ms_per_step"] = round(e["ms_per_step"] + float(d_ms), 4)
        for d in dsts:
            m.seq_free(d)
        # the shared-prefix form of the fork: full pages by reference, and
        # the batched steps' attention over the prefix runs once for all
        # branches (cascade attention)
        dsts = [m.seq_create() for _ in range(B)]
        m.kv_fork(src, dsts, shared=True)
        m.generate(dsts, start, 2)  # capture the cascade graph outside the timing
        for d in dsts:
            m.seq_free(d)
        dsts = [m.seq_create() for _ in range(B)]
        t_fork_sh = _events(torch, stream, lambda: m.kv_fork(src, dsts, shared=True))
        t_dec_sh = _events(torch, stream, lambda: m.generate(dsts, start, D))
        kms, kk = m.profile_batch(dsts, start, [m.seq_length(d) for d in dsts])
        per_kind_sh = {}
        for d_ms, k in zip(kms, kk):
            e = per_kind_sh.setdefault(KIND_NAMES.get(int(k), str(int(k))), {"launches_per_step": 0,
                                                                              "ms_per_step": 0.0})
            e["launches_per_step"] += 1
            e["ms_per_step"] = round(e["ms_per_step"] + float(d_ms), 4)
        for d in dsts:
            m.seq_free(d)
        m.seq_free(src)
        # the same branches from 8 independent prefills
        t_ind = 0.0
        seqs = []
        for b in range(B):
            q = m.seq_create()
            t_ind += _events(torch, stream, lambda: m.prefill(q, prefix))
            seqs.append(q)
    kv_bytes = cfg.n_layers * 2 * P * cfg.kv_dim * 2
    fork_path = t_pre + t_fork + t_dec
    shared_path = t_pre + t_fork_sh + t_dec_sh
    indep_path = t_ind + t_dec
    m.close()
    return base_line("shared-prefix fork: branch tokens/s of prefill + fork + batch-8 decode, 8B-shape Q4_0",
                     B * D / fork_path, "tok/s", D, 2, 1000 * t_dec / D,
                     f"fork8b: prefix {P} -> {B} branches x {D} greedy tokens, batch {B}",
                     {"fork": {"prefill_ms": round(1000 * t_pre, 2), "prefill_tok_s": round(P / t_pre, 1),
                               "fork_ms": round(1000 * t_fork, 3),
                               "fork_copy_gbs": round(2 * B * kv_bytes / t_fork / 1e9, 1),
                               "decode_ms": round(1000 * t_dec, 2), "decode_tok_s": round(B * D / t_dec, 1),
                               "fork_path_s": round(fork_path, 4), "independent_prefills_path_s": round(indep_path, 4),
                               "speedup_vs_independent": round(indep_path / fork_path, 3),
                               "shared_pages": {"fork_ms": round(1000 * t_fork_sh, 3),
                                                "decode_ms": round(1000 * t_dec_sh, 2),
                                                "decode_tok_s": round(B * D / t_dec_sh, 1),
                                                "fork_path_s": round(shared_path, 4),
                                                "speedup_vs_independent": round(indep_path / shared_path, 3),
                                                "kernels": per_kind_sh}},
                      "kernels": per_kind, "clocks": clk.summary()})


def run_skip(args):
    """Decode with layer skip (the engine page's calibration): after a --ctx
    prefill, one decode step measures every layer's output/input cosine;
    the layers above the threshold are skipped and greedy decode is timed
    with and without the skips."""
    import torch
    import synth
    from decode_llama_step_gb300 import dls
    cfg = load_config(args.config, args.layers)
    D, W = args.steps, max(args.warmup, 1)
    w = synth.model_weights(cfg)
    stream = torch.cuda.Stream()
    m = dls.Model(cfg, w, max_seqs=1, max_ctx=args.ctx + 2 * (D + W) + 8, stream=stream)
    del w
    seq = m.seq_create()
    prompt = synth.prompt_tokens(cfg, args.ctx, seed=1)
    lg = torch.empty(cfg.vocab, device="cuda")
    m.prefill(seq, prompt, lg)
    tok = int(torch.argmax(lg).item())
    cos = m.layer_cosines(seq, tok, args.ctx)
    mask = cos > args.skip_threshold
    tok = int(m.generate([seq], [tok], W)[-1, 0])
    t_full = _events(torch, stream, lambda: m.generate([seq], [tok], D))
    m.set_layer_skip(mask)
    tok = int(m.generate([seq], [tok], W)[-1, 0])
    with ClockSampler(0) as clk:
        t_skip = _events(torch, stream, lambda: m.generate([seq], [tok], D))
    m.close()
    return base_line(f"decode tok/s with layer skip (calibrated cosine > {args.skip_threshold}), "
                     f"{cfg.name}-shape {'Q8_0' if cfg.wtype == 8 else 'Q4_0'} batch 1",
                     D / t_skip, "tok/s", D, W, 1000 * t_skip / D,
                     f"{cfg.name} batch-1 greedy decode after a {args.ctx}-token prefill, layers skipped by calibration",
                     {"skip": {"threshold": args.skip_threshold, "n_skipped": int(mask.sum()),
                               "skipped_layers": [int(i) for i in np.nonzero(mask)[0]],
                               "cosines": [round(float(c), 5) for c in cos],
                               "tok_s_all_layers": round(D / t_full, 2), "tok_s_with_skip": round(D / t_skip, 2),
                               "speedup": round(t_full / t_skip, 3)},
                      "clocks": clk.summary()})


def run_spec(args):
    """Self-speculative greedy decoding against plain greedy decoding from the
    same state (a copy of one prefilled sequence for every run).  --config
    70b: 70B Q4_0 under the 24 GB device budget, and the draft is the
    resident layers (the streamed ones are skipped, so draft steps copy
    nothing in); other configs: all layers resident, and the draft skips the
    layers whose calibrated cosine exceeds --skip-threshold."""
    import torch
    import synth
    from decode_llama_step_gb300 import dls
    cfg = load_config(args.config, args.layers)
    streamed = cfg.name == "70b"
    ctx = (args.ctx if args.ctx != 2048 else cfg.workload["ctx"]) if streamed else args.ctx
    D = args.steps
    ks = [int(k) for k in args.draft_k.split(",") if k.strip()]
    w = synth.model_weights(cfg)
    stream = torch.cuda.Stream()
    budget = cfg.workload["budget_bytes"] if streamed else 0
    m = dls.Model(cfg, w, max_seqs=2, max_ctx=ctx + D + 64, stream=stream, device_budget_bytes=budget)
    del w
    base, work = m.seq_create(), m.seq_create()
    prompt = synth.prompt_tokens(cfg, ctx, seed=1)
    lg = torch.empty(cfg.vocab, device="cuda")
    m.prefill(base, prompt, lg)
    tok = int(torch.argmax(lg).item())
    if streamed:
        res = m.resident_layers()
        mask = np.array([l >= res for l in range(cfg.n_layers)])
        draft = f"the {res} resident layers ({cfg.n_layers - res} streamed layers skipped)"
    else:
        m.kv_fork(base, [work])
        cos = m.layer_cosines(work, tok, ctx)
        mask = cos > args.skip_threshold
        draft = f"{cfg.n_layers - int(mask.sum())} layers (cosine > {args.skip_threshold} skipped: " \
                f"{[int(i) for i in np.nonzero(mask)[0]]})"
    m.kv_fork(base, [work])
    m.generate([work], [tok], max(args.warmup, 1))
    m.kv_fork(base, [work])
    with ClockSampler(0) as clk:
        t_plain = _events(torch, stream, lambda: m.generate([work], [tok], D))
    m.kv_fork(base, [work])
    ref = m.generate([work], [tok], D)[:, 0]
    runs = {}
    best = None
    for k in ks:
        m.kv_fork(base, [work])
        m.generate_speculative(work, tok, min(D, 8), mask, k)   # warm-up: graphs, pages
        m.kv_fork(base, [work])
        out = {}

        def go():
            out["r"] = m.generate_speculative(work, tok, D, mask, k)
        t = _events(torch, stream, go)
        toks, st = out["r"]
        same = int(np.argmax(np.concatenate([toks != ref, [True]])))
        runs[f"k={k}"] = {"tok_s": round(D / t, 3), "ms_per_token": round(1000 * t / D, 3),
                          "speedup": round(t_plain / t, 3), "rounds": st["rounds"], "drafted": st["drafted"],
                          "accepted": st["accepted"],
                          "acceptance": round(st["accepted"] / max(st["drafted"], 1), 4),
                          "tokens_per_round": round(D / st["rounds"], 3),
                          "tokens_equal_to_plain_greedy": same}
        if best is None or D / t > best[1]:
            best = (k, D / t, t)
    m.close()
    k, v, t = best
    return base_line(f"self-speculative greedy decode tok/s, {cfg.name}-shape "
                     f"{'Q8_0' if cfg.wtype == 8 else 'Q4_0'} batch 1"
                     + (", 24 GB device budget (layer streaming)" if streamed else ""),
                     v, "tok/s", D, args.warmup, 1000 * t / D,
                     f"{cfg.name} greedy decode of {D} tokens after a {ctx}-token prompt; draft = {draft}; "
                     f"best draft length k={k}",
                     {"speculative": {"plain_tok_s": round(D / t_plain, 3), "runs": runs, "draft": draft},
                      "clocks": clk.summary()})


KQ_SHAPES_70B = {"wq/wo": (8192, 8192), "wk/wv": (1024, 8192), "w_gate/w_up": (28672, 8192),
                 "w_down": (8192, 28672)}
# Q4_K_M's usual type per 70B matrix (the attention value and FFN down
# projections kept at 6 bits, the rest at 4)
KQ_Q4_K_M = {"wq": "q4_k", "wk": "q4_k", "wv": "q6_k", "wo": "q4_k", "w_gate": "q4_k", "w_up": "q4_k",
             "w_down": "q6_k"}


def run_kquant(args):
    """K-quant dequant-GEMV bandwidth on the 70B projection shapes: each
    (format, shape) timed over --steps launches that cycle through enough
    copies of the matrix to exceed the L2 several times (every launch reads
    its weights from HBM)."""
    import torch
    import synth
    from decode_llama_step_gb300 import dls
    peak, src = peaks()
    stream = torch.cuda.Stream()
    L2 = 129 * 2 ** 20
    res = {}
    with ClockSampler(0) as clk:
        for fmt in ("q4_k", "q5_k", "q6_k"):
            for name, (rows, cols) in KQ_SHAPES_70B.items():
                if args.kq_only and args.kq_only != f"{fmt}:{rows}x{cols}":
                    continue
                blocks = torch.from_numpy(synth.kquant_matrix(synth.stream_key("bench-kq", fmt, name), rows, cols,
                                                              fmt)).cuda()
                nbytes = dls.kquant_packed_bytes(fmt, rows, cols)
                copies = max(2, -(-4 * L2 // nbytes))
                packed = [torch.empty(nbytes, dtype=torch.uint8, device="cuda") for _ in range(copies)]
                for p_ in packed:
                    dls.kquant_pack(fmt, blocks, rows, cols, p_, stream=stream)
                del blocks
                x = torch.randn(cols, device="cuda")
                y = torch.empty(rows, device="cuda")
                status = torch.zeros(1, dtype=torch.int32, device="cuda")
                for i in range(max(args.warmup, 3)):
                    dls.kquant_gemv(fmt, packed[i % copies], rows, cols, x, y, status, stream)
                n = max(args.steps, copies)

                def go():
                    for i in range(n):
                        dls.kquant_gemv(fmt, packed[i % copies], rows, cols, x, y, status, stream)
                t = _events(torch, stream, go) / n
                assert int(status.item()) == 0
                alg = dls.kquant_packed_bytes(fmt, rows, cols) + 4 * (rows + cols)
                res[f"{fmt} {name} {rows}x{cols}"] = {"us": round(1e6 * t, 2), "bytes": alg,
                                                      "gbs": round(alg / t / 1e9, 1),
                                                      "frac": round(alg / t / 1e9 / peak, 4)}
                del packed
    if args.kq_only:
        (key, r), = res.items()
        return base_line(f"{key} dequant-GEMV GB/s", r["gbs"], "GB/s", args.steps, args.warmup, r["us"] / 1000.0,
                         f"one K-quant GEMV shape ({key}), batch 1, inputs > L2", {"kquant": res})
    layer_us = sum(res[f"{KQ_Q4_K_M[m]} {k} {KQ_SHAPES_70B[k][0]}x{KQ_SHAPES_70B[k][1]}"]["us"]
                   for k in KQ_SHAPES_70B for m in k.split("/"))
    layer_bytes = sum(res[f"{KQ_Q4_K_M[m]} {k} {KQ_SHAPES_70B[k][0]}x{KQ_SHAPES_70B[k][1]}"]["bytes"]
                      for k in KQ_SHAPES_70B for m in k.split("/"))
    top = res["q4_k w_gate/w_up 28672x8192"]
    return base_line("Q4_K dequant-GEMV GB/s, 70B gate/up shape (28672 x 8192)", top["gbs"], "GB/s", args.steps,
                     args.warmup, top["us"] / 1000.0, "70B projection shapes, Q4_K and Q6_K, batch 1, inputs > L2",
                     {"roofline": {"bound": "hbm", "achieved": top["gbs"], "peak": peak, "unit": "GB/s",
                                   "frac": top["frac"], "traffic": None, "peak_source": src},
                      "kquant": res,
                      "q4_k_m_layer": {"matrices": KQ_Q4_K_M, "gemv_us_sum": round(layer_us, 1),
                                       "bytes": layer_bytes,
                                       "gbs": round(layer_bytes / (layer_us * 1e-6) / 1e9, 1),
                                       "how": "sum of the seven matrices' measured GEMV times"},
                      "clocks": clk.summary()})


def run_batch(args):
    """Batched decode of 2, 4 and 8 sequences (copies of one --ctx prompt's
    cache): greedy tok/s over --steps graph-replayed steps per batch size,
    and one step's kernels timed one by one.  DLS_BATCH_GEMM (tc or rg)
    forces one projection path for every batch size."""
    import torch
    import synth
    from decode_llama_step_gb300 import dls
    cfg = load_config(args.config, args.layers)
    D, W = args.steps, max(args.warmup, 1)
    w = synth.model_weights(cfg)
    stream = torch.cuda.Stream()
    m = dls.Model(cfg, w, max_seqs=9, max_ctx=args.ctx + D + W + 8, max_batch=8, page_tokens=64, stream=stream)
    del w
    base = m.seq_create()
    m.prefill(base, synth.prompt_tokens(cfg, args.ctx, seed=1))
    res = {}
    with ClockSampler(0) as clk:
        for n in (2, 4, 8):
            seqs = [m.seq_create() for _ in range(n)]
            m.kv_fork(base, seqs)
            toks = [100 + i for i in range(n)]
            m.generate(seqs, toks, W)
            t = _events(torch, stream, lambda: m.generate(seqs, toks, D))
            kms, kk = m.profile_batch(seqs, toks, [m.seq_length(s) for s in seqs])
            per_kind = {}
            for d_ms, k in zip(kms, kk):
                name = KIND_NAMES.get(int(k), str(int(k)))
                per_kind[name] = round(per_kind.get(name, 0.0) + float(d_ms), 4)
            res[f"batch{n}"] = {"tok_s": round(n * D / t, 1), "ms_per_step": round(1000 * t / D, 3),
                                "kernels_ms": per_kind, "kernels_total_ms": round(sum(per_kind.values()), 3)}
            for s_ in seqs:
                m.seq_free(s_)
    m.close()
    b = res["batch8"]
    path = os.environ.get("DLS_BATCH_GEMM", "default (rows <= 4: multi-row GEMV; 5-8: tensor-core GEMM)")
    return base_line(f"batched decode tok/s, {cfg.name}-shape {'Q8_0' if cfg.wtype == 8 else 'Q4_0'}, batch 8",
                     b["tok_s"], "tok/s", D, W, b["ms_per_step"],
                     f"{cfg.name} batched greedy decode of copies of a {args.ctx}-token cache, batch 2/4/8",
                     {"batch": res, "projection_path": path, "clocks": clk.summary()})


def h2d_peak(torch, chunk=256 << 20, inflight=4, reps=10):
    """Best pinned host -> device copy rate over several methods: 256 MB
    chunks, four in flight, issued on one, two or four streams (copy
    engines), and the library's SM-driven copy kernel (CTAs reading the
    pinned buffer over the host link) at several CTA counts.  Returns
    (best GB/s, {method: GB/s})."""
    from decode_llama_step_gb300 import dls
    host = torch.empty(chunk * inflight, dtype=torch.uint8, pin_memory=True)
    host.fill_(1)
    dev = torch.empty(chunk * inflight, dtype=torch.uint8, device="cuda")
    main = torch.cuda.Stream()
    rates = {}
    for ns in (1, 2, 4):
        streams = [torch.cuda.Stream() for _ in range(ns)]
        best = 0.0
        for _ in range(reps):
            def go():
                ev = torch.cuda.Event()
                ev.record(main)
                for i in range(inflight):
                    st = streams[i % ns]
                    st.wait_event(ev)
                    with torch.cuda.stream(st):
                        dev[i * chunk:(i + 1) * chunk].copy_(host[i * chunk:(i + 1) * chunk], non_blocking=True)
                for st in streams:
                    e2 = torch.cuda.Event()
                    e2.record(st)
                    main.wait_event(e2)
            t = _events(torch, main, go)
            best = max(best, chunk * inflight / t / 1e9)
        rates[f"copy_engines_{ns}_streams"] = round(best, 1)
    for ctas in (16, 32, 64, 152):
        best = 0.0
        for _ in range(reps):
            t = _events(torch, main, lambda: dls.h2d_copy_sm(dev, host, chunk * inflight, ctas, main))
            best = max(best, chunk * inflight / t / 1e9)
        rates[f"sm_kernel_{ctas}_ctas"] = round(best, 1)
    torch.cuda.synchronize()
    assert torch.equal(dev[:4096].cpu(), host[:4096])
    return max(rates.values()), rates


def run_kmodel(args):
    """The 70B shape as a Q4_K_M-style file (value and down projections and
    the LM head Q6_K, everything else Q4_K): decode through the mixed-format
    path, resident and under the 24 GB device budget, after a --ctx prompt
    (default 64 here: prefill of a mixed model runs 8 tokens per pass)."""
    import torch
    import synth
    from decode_llama_step_gb300 import dls
    cfg = load_config("70b", args.layers)
    ctx = args.ctx if args.ctx != 2048 else 64
    D = min(args.steps, 32)
    t0 = time.time()
    w = synth.model_weights_k(cfg, synth.Q4_K_M)
    gen_s = time.time() - t0
    stream = torch.cuda.Stream()
    prompt = synth.prompt_tokens(cfg, ctx, seed=1)
    out = {}
    for label, budget in (("resident", 0), ("budget_24GB", cfg.workload["budget_bytes"])):
        m = dls.Model(cfg, w, max_seqs=1, max_ctx=ctx + D + 16, stream=stream, device_budget_bytes=budget)
        s = m.seq_create()
        t_pre = _events(torch, stream, lambda: m.prefill(s, prompt))
        m.generate([s], [1], 2)
        with ClockSampler(0) as clk:
            t = _events(torch, stream, lambda: m.generate([s], [1], D))
        res = m.resident_layers()
        lb = m.layer_bytes()
        weight_bytes = cfg.n_layers * lb
        streamed = (cfg.n_layers - res) * lb
        out[label] = {"resident_layers": res, "decode_tok_s": round(D / t, 3), "ms_per_token": round(1000 * t / D, 2),
                      "prefill_s": round(t_pre, 2), "layer_bytes": lb,
                      "hbm_gbs_layers": round((weight_bytes - streamed) / (t / D) / 1e9, 1),
                      "h2d_gbs": round(streamed / (t / D) / 1e9, 1) if streamed else None,
                      "clocks": clk.summary()}
        m.close()
    del w
    r = out["resident"]
    return base_line("70B-shape Q4_K_M-style decode tok/s (resident)", r["decode_tok_s"], "tok/s", D, 2,
                     r["ms_per_token"], f"70b Q4_K_M-style (Q4_K + Q6_K), KV ctx {ctx}, {D} greedy tokens",
                     {"kquant_model": out, "weights_gen_s": round(gen_s, 1),
                      "context_note": "the engine page quotes 0.3 tok/s for 70B Q4_K_M on an RTX 3090 with "
                                      "tiered caching (context, not a target)"})


def run_h2d(args):
    """Host -> device bandwidth only: the methods h2d_peak compares."""
    import torch
    peak, rates = h2d_peak(torch)
    return base_line("pinned host -> device copy GB/s (best method)", peak, "GB/s", 10, 1, 0.0,
                     "4 x 256 MB pinned host buffers to device memory", {"h2d_rates_gbs": rates})


def run_stream(args):
    """70B Q4_0 decode at KV length --ctx (default 4096): all layers resident
    vs a 24 GB device budget (the layers that do not fit stream from pinned
    host memory through two device buffers)."""
    import torch
    import synth
    from decode_llama_step_gb300 import dls
    cfg = synth.get_config("70b")
    ctx = args.ctx if args.ctx != 2048 else cfg.workload["ctx"]
    D = min(args.steps, cfg.workload["decode"])
    w = synth.model_weights(cfg)
    stream = torch.cuda.Stream()
    peak_h2d, h2d_rates = h2d_peak(torch)
    prompt = synth.prompt_tokens(cfg, ctx, seed=1)
    out = {}
    sm_best = max((k for k in h2d_rates if k.startswith("sm_kernel")), key=lambda k: h2d_rates[k])
    sm_ctas = int(sm_best.split("_")[2])
    runs = [("resident", 0, None), ("budget_24GB", cfg.workload["budget_bytes"], None),
            ("budget_24GB_sm_copy", cfg.workload["budget_bytes"], f"sm:{sm_ctas}")]
    for label, budget, copy_mode in runs:
        if copy_mode:
            os.environ["DLS_STREAM_COPY"] = copy_mode      # read when the model is created
        try:
            m = dls.Model(cfg, w, max_seqs=1, max_ctx=ctx + D + 16, stream=stream, device_budget_bytes=budget)
        finally:
            os.environ.pop("DLS_STREAM_COPY", None)
        s = m.seq_create()
        t_pre = _events(torch, stream, lambda: m.prefill(s, prompt))
        m.generate([s], [1], 2)
        with ClockSampler(0) as clk:
            t = _events(torch, stream, lambda: m.generate([s], [1], D))
        res = m.resident_layers()
        streamed_bytes = (cfg.n_layers - res) * m.layer_bytes()
        out[label] = {"resident_layers": res, "decode_tok_s": round(D / t, 3), "ms_per_token": round(1000 * t / D, 2),
                      "prefill_s": round(t_pre, 2), "h2d_bytes_per_token": streamed_bytes,
                      "h2d_gbs": round(streamed_bytes / (t / D) / 1e9, 1) if streamed_bytes else None,
                      "h2d_frac_of_peak": round(streamed_bytes / (t / D) / 1e9 / peak_h2d, 4) if streamed_bytes else None,
                      "clocks": clk.summary(), "copy": copy_mode or "copy engines (cudaMemcpyAsync)"}
        m.close()
    del w
    b = max((out["budget_24GB"], out["budget_24GB_sm_copy"]), key=lambda r: r["decode_tok_s"])
    return base_line("70B-shape Q4_0 decode tok/s with a 24 GB device budget (layer streaming)", b["decode_tok_s"],
                     "tok/s", D, 2, b["ms_per_token"], f"70b Q4_0, KV ctx {ctx}, {D} greedy tokens",
                     {"stream": out, "h2d_peak_gbs": round(peak_h2d, 1), "h2d_rates_gbs": h2d_rates,
                      "h2d_peak_how": "best of: pinned cudaMemcpyAsync of 4 x 256 MB on 1, 2 or 4 streams; the "
                                      "SM-driven copy kernel at 16-152 CTAs; best of 10 each"})


def gemv_bytes(rows, cols, wtype):
    nb = (cols + 31) // 32
    per_block = 34 if wtype == 8 else 18
    return rows * nb * per_block + cols * 4 + rows * 4


def step_bytes(cfg, ctx_len):
    """Algorithmic HBM bytes of one decode token at KV length ctx_len."""
    H, F, V = cfg.hidden, cfg.ffn, cfg.vocab
    qd, kvd = cfg.q_dim, cfg.kv_dim
    per_layer = (gemv_bytes(qd + 2 * kvd, H, cfg.wtype) + gemv_bytes(H, qd, cfg.wtype)
                 + gemv_bytes(2 * F, H, cfg.wtype) + gemv_bytes(H, F, cfg.wtype)
                 + 2 * ctx_len * kvd * 2)            # K and V read (fp16)
    head = gemv_bytes(V, H, cfg.wtype)
    return cfg.n_layers * per_layer + head


def kind_bytes(cfg, kind, ctx_len):
    H, F, V = cfg.hidden, cfg.ffn, cfg.vocab
    qd, kvd = cfg.q_dim, cfg.kv_dim
    return {2: gemv_bytes(qd + 2 * kvd, H, cfg.wtype) + 2 * kvd * 2,
            3: 2 * ctx_len * kvd * 2 + 2 * qd * 4,
            4: gemv_bytes(H, qd, cfg.wtype),
            5: gemv_bytes(2 * F, H, cfg.wtype),
            6: gemv_bytes(H, F, cfg.wtype) + F * 4,
            7: gemv_bytes(V, H, cfg.wtype)}.get(kind, 0)


class ClockSampler:
    """nvidia-smi samples (every 200 ms) while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.tmp,
                                         stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        self.tmp.flush()
        self.tmp.seek(0)
        sm, mx, reasons = [], None, set()
        for line in self.tmp.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def cpu_oracle_sample(cfg, ctx, n_layer_samples=2):
    """Time the fp64 oracle's decode step on a bounded sample: n layers of the
    model at KV length ctx (seeded fp16-valued cache) plus the LM head, scaled
    to the whole model.  Returns (tok/s, seconds, description, cores)."""
    import synth
    from oracle import OracleModel, ops

    layers = list(range(n_layer_samples))
    w = synth.model_weights(cfg, layers=layers)
    orc = OracleModel(cfg, w, cache_bytes=0)
    seq = orc.new_seq(capacity=ctx + 1)
    for l in layers:
        k = ops.round_f16(synth.normal(synth.stream_key("bench-kv", l, "k"), ctx * cfg.kv_dim, 1.0))
        v = ops.round_f16(synth.normal(synth.stream_key("bench-kv", l, "v"), ctx * cfg.kv_dim, 1.0))
        seq.set_layer(l, k.reshape(ctx, cfg.n_kv_heads, cfg.head_dim), v.reshape(ctx, cfg.n_kv_heads, cfg.head_dim))
    x = orc.embed(1)
    t0 = time.perf_counter()
    for l in layers:
        x = orc.layer_forward(l, x, ctx, seq)
    t_layers = (time.perf_counter() - t0) / len(layers)
    t1 = time.perf_counter()
    orc.final_logits(x)
    t_head = time.perf_counter() - t1
    per_tok = t_layers * cfg.n_layers + t_head
    cores = len(os.sched_getaffinity(0))
    desc = (f"fp64 oracle decode of layers 0-{len(layers) - 1} of {cfg.n_layers} at KV length {ctx} plus the "
            f"LM head, scaled to {cfg.n_layers} layers ({t_layers:.2f} s/layer, head {t_head:.2f} s)")
    return 1.0 / per_tok, t_layers * len(layers) + t_head, desc, cores


def cpu_oracle_prefill_sample(cfg, T):
    """Time the fp64 oracle's prefill on a bounded sample: layer 0 of the
    model over the whole T-token prompt plus the last token's LM head,
    scaled to the whole model.  Returns (tok/s, description, cores)."""
    import synth
    from oracle import OracleModel

    w = synth.model_weights(cfg, layers=[0])
    orc = OracleModel(cfg, w, cache_bytes=0)
    seq = orc.new_seq(capacity=T + 1)
    X = orc.embed(synth.prompt_tokens(cfg, T, seed=1))
    t0 = time.perf_counter()
    X = orc.layer_forward(0, X, 0, seq)
    t_layer = time.perf_counter() - t0
    t1 = time.perf_counter()
    orc.final_logits(X[-1])
    t_head = time.perf_counter() - t1
    per_prefill = t_layer * cfg.n_layers + t_head
    cores = len(os.sched_getaffinity(0))
    desc = (f"fp64 oracle prefill of layer 0 of {cfg.n_layers} over the {T}-token prompt plus the LM head, scaled "
            f"to {cfg.n_layers} layers ({t_layer:.2f} s/layer, head {t_head:.2f} s)")
    return T / per_prefill, desc, cores


def run_reference(args):
    """The reference arm: the fp64 oracle on the host cores, on the headline
    workload.  Each step is a bounded sample of a decode step: one layer of
    the 8B model (alternating between two layers) at KV length --ctx, run as
    the oracle runs it; --warmup untimed steps, then --steps timed ones.  The
    LM head is timed once.  tok/s = 1 / (n_layers x mean layer time + head)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import synth
    from oracle import OracleModel, ops
    cfg = synth.get_config(args.config)
    K, W, ctx = max(1, args.steps), max(0, args.warmup), args.ctx
    layers = [0, 1]
    w = synth.model_weights(cfg, layers=layers)
    orc = OracleModel(cfg, w, cache_bytes=0)
    seq = orc.new_seq(capacity=ctx + 1)
    for l in layers:
        k = ops.round_f16(synth.normal(synth.stream_key("bench-kv", l, "k"), ctx * cfg.kv_dim, 1.0))
        v = ops.round_f16(synth.normal(synth.stream_key("bench-kv", l, "v"), ctx * cfg.kv_dim, 1.0))
        seq.set_layer(l, k.reshape(ctx, cfg.n_kv_heads, cfg.head_dim), v.reshape(ctx, cfg.n_kv_heads, cfg.head_dim))
    x = orc.embed(1)

    def step(i):
        orc.layer_forward(layers[i % len(layers)], x, ctx, seq)
        seq.truncate(ctx)   # the next sample appends at the same position

    for i in range(W):
        step(i)
    t0 = time.perf_counter()
    for i in range(K):
        step(W + i)
    t_layer = (time.perf_counter() - t0) / K
    t1 = time.perf_counter()
    orc.final_logits(x)
    t_head = time.perf_counter() - t1
    per_tok = t_layer * cfg.n_layers + t_head
    tps = 1.0 / per_tok
    cores = len(os.sched_getaffinity(0))
    desc = (f"fp64 oracle: {K} timed steps (after {W} untimed), each one layer of {cfg.n_layers} (layers 0 and 1 "
            f"alternating) at KV length {ctx}; LM head once; {t_layer:.3f} s/layer, head {t_head:.2f} s, scaled to "
            f"{cfg.n_layers} layers")
    line = {"metric": METRIC, "impl": "reference", "value": round(tps, 6), "unit": "tok/s", "n_gpus": args.gpus,
            "steps": K, "warmup": W, "ms_per_step": round(1000.0 * per_tok, 3), "higher_is_better": True,
            "step_kind": f"one timed step = one layer of the {cfg.n_layers}-layer decode step (a bounded sample); "
                         f"ms_per_step and value are the per-token figures scaled from the samples",
            "ms_per_sample": round(1000.0 * t_layer, 3), "ms_lm_head": round(1000.0 * t_head, 3),
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{cfg.name} Q8_0 batch-1 greedy decode, KV ctx {ctx}", "ctx": ctx, "batch": 1},
            "cpu_baseline": {"value": round(tps, 6), "unit": "tok/s", "cores": cores, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": round(tps, 6), "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    if args.workload != "decode":
        if int(os.environ.get("RANK", "0")) != 0:
            return 0
        fn = {"prefill": run_prefill, "fork": run_fork, "stream": run_stream, "skip": run_skip,
              "spec": run_spec, "kquant": run_kquant, "batch": run_batch, "h2d": run_h2d,
              "kmodel": run_kmodel}[args.workload]
        print(json.dumps(fn(args)), flush=True)
        return 0

    import torch

    import synth
    from decode_llama_step_gb300 import dls

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    cfg = load_config(args.config, args.layers)
    t0 = time.time()
    w = synth.model_weights(cfg)
    gen_s = time.time() - t0
    stream = torch.cuda.Stream()
    extra = args.warmup + args.steps + args.e2e_steps + args.profile_steps + 8
    t0 = time.time()
    m = dls.Model(cfg, w, max_seqs=1, max_ctx=args.ctx + extra, stream=stream)
    create_s = time.time() - t0
    del w
    seq = m.seq_create()
    prompt = synth.prompt_tokens(cfg, args.ctx, seed=1)
    logits = torch.empty(cfg.vocab, device="cuda")
    t0 = time.time()
    m.prefill(seq, prompt, logits)
    prefill_s = time.time() - t0
    tok = int(torch.argmax(logits).item())

    # warm-up (also captures the generation graph)
    toks = m.generate([seq], [tok], args.warmup)
    tok = int(toks[-1, 0])
    ctx0 = m.seq_length(seq)

    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        if args.profile_region:
            torch.cuda.profiler.start()
        start.record(stream)
        toks = m.generate([seq], [tok], args.steps)
        end.record(stream)
        end.synchronize()
        if args.profile_region:
            torch.cuda.profiler.stop()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    ms = max_over_ranks(start.elapsed_time(end), dist, "cuda")
    ms_per_step = ms / args.steps
    value = replica_throughput(world, args.steps, ms)
    tok = int(toks[-1, 0])
    launches = m.launches_per_step()

    # roofline: per-kernel device times from event-instrumented steps
    kinds_ms = {}
    pos = m.seq_length(seq)
    for _ in range(args.profile_steps):
        kms, kk = m.profile_step(seq, tok, pos)
        pos += 1
        for d, k in zip(kms, kk):
            kinds_ms.setdefault(int(k), []).append(float(d))
    ctx_mid = ctx0 + args.steps // 2
    ctx_prof = pos - args.profile_steps // 2  # mean KV length of the profiled steps
    gemv_kinds = (2, 4, 5, 6, 7)
    gemv_bytes_total = sum(kind_bytes(cfg, k, ctx_mid) * len(kinds_ms.get(k, [])) for k in gemv_kinds)
    gemv_ms_total = sum(sum(kinds_ms.get(k, [])) for k in gemv_kinds)
    gemv_launches = sum(len(kinds_ms.get(k, [])) for k in gemv_kinds)
    peak, peak_src = peaks()
    achieved = gemv_bytes_total / (gemv_ms_total / 1000.0) / 1e9 if gemv_ms_total else 0.0
    persistent = launches == 1
    step_used, step_why = m.step_kernel_in_use()
    if persistent:
        # one cooperative launch per token: the step kernel is the whole
        # step; its duration is the span of its phase timestamps
        kern_ms = sum(sum(v) for v in kinds_ms.values()) / max(args.profile_steps, 1)
        kern_b = step_bytes(cfg, ctx_prof)
        src = "step.cu"
        achieved = kern_b / (kern_ms / 1000.0) / 1e9 if kern_ms else 0.0
        kern = {"kernel": "persistent decode-step kernel (embedding, 32 layers, LM head, greedy pick in one launch)",
                "bytes_per_launch": kern_b, "avg_launch_us": round(1000.0 * kern_ms, 2)}
    else:
        src = "gemv.cu"
        kern = {"kernel": "dequant-GEMV (QKV, O, gate/up, down, LM head launches of one step)",
                "bytes_per_launch": round(gemv_bytes_total / max(gemv_launches, 1)),
                "avg_launch_us": round(1000.0 * gemv_ms_total / max(gemv_launches, 1), 2)}
    src_sha = hashlib.sha256(open(os.path.join(ROOT, "decode_llama_step_gb300", "csrc", src), "rb").read()).hexdigest()[:16]
    nt = NCU_TRAFFIC.get(src_sha)
    traffic = round(nt["ratio"] * kern["bytes_per_launch"]) if nt else None
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": traffic, **kern,
                "peak_source": f"{peak_src} (MEMORY copy, hbm_gbs)"}
    step_b = step_bytes(cfg, ctx_mid)
    whole = step_b / (ms_per_step / 1000.0) / 1e9
    per_kind = {KIND_NAMES.get(k, str(k)): {"launches_per_step": len(v) // max(args.profile_steps, 1),
                                            "ms_per_step": round(sum(v) / max(args.profile_steps, 1), 4)}
                for k, v in sorted(kinds_ms.items())}

    # end to end: host token in, host logits out (pinned), host argmax, per step
    host_logits = torch.empty(cfg.vocab, dtype=torch.float32, pin_memory=True)
    hl = host_logits.numpy()
    e2e_n = args.e2e_steps
    pos = m.seq_length(seq)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(e2e_n):
        m.decode_step(seq, tok, pos + i, host_logits)
        tok = int(np.argmax(hl))
    e2e_s = time.perf_counter() - t0
    e2e_val = world * e2e_n / e2e_s

    line = {"metric": METRIC, "value": round(value, 3), "unit": "tok/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int32+f32", "data": "synthetic",
            "arith": "Q8_0 codes x int16-quantised activation slices (16 per lane), exact int32 dot products, fp32 "
                     "scaling and accumulation; fp16 KV cache, fp32 attention",
            "config": {"workload": f"{cfg.name}-shape {'Q8_0' if cfg.wtype == 8 else 'Q4_0'} batch-1 greedy decode, "
                                   f"{cfg.n_layers} layers, KV ctx {ctx0}..{ctx0 + args.steps}",
                       "ctx": args.ctx, "batch": 1, "weights": "seeded N(0,0.02), quantised Q8_0",
                       "l2": "no flush: 8.2 GB of weights per step > 126 MB L2",
                       "parallelism": f"replicas x{world}"},
            "hbm": {"algorithmic_bytes_per_step": step_b, "achieved_gbs": round(whole, 1),
                    "frac_of_peak": round(whole / peak, 4), "peak_gbs": peak},
            "roofline": roofline,
            "decode_path": "persistent step kernel" if step_used else f"separate kernels ({step_why})",
            "kernels": per_kind,
            "e2e": {"value": round(e2e_val, 3), "unit": "tok/s", "h2d_bytes_per_step": 8,
                    "d2h_bytes_per_step": cfg.vocab * 4,
                    "how": "dls_decode_step with host token, pinned host logits, host argmax"},
            "gpu_launches": launches * args.steps,
            "clocks": clk.summary(),
            "setup_s": {"weights": round(gen_s, 1), "create": round(create_s, 1), "prefill": round(prefill_s, 2),
                        "prefill_tok_s": round(args.ctx / prefill_s, 1)}}
    if rank == 0 and not args.no_cpu_baseline:
        tps, secs, desc, cores = cpu_oracle_sample(cfg, args.ctx)
        line["cpu_baseline"] = {"value": round(tps, 6), "unit": "tok/s", "cores": cores, "kind": "oracle",
                                "sample": desc}
    m.close()
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
