"""Benchmark of the MLA latent-KV decode hot path on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

A step is one pass of the hot path over one batch: mla_absorb_q -> mla_decode (split-K
attention + log-sum-exp combine) -> mla_out, on the DeepSeek-V2-shaped decode batch
(B=16, 4096 cached tokens each, 128 heads, d_c=512, d_rope=64, page size 64, shuffled pages).
Inputs are synthetic and resident in HBM; L2 is flushed between steps (a 256 MB write, then
read back, so that no dirty lines of the flush remain).
With --gpus N > 1 (launched by torchrun) every rank runs an independent replica (the path
shards by sequence with no exchange), and value is the job total.

--impl reference times the CPU float64 oracle on bounded samples of the same workload.
Prints one JSON line.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import mla_workloads as W  # noqa: E402

METRIC = "MLA decode tokens/s, HBM GB/s and % of roofline (B=16, T=4096, 128 heads)"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6400.0
FALLBACK_BF16_TFLOPS = 1800.0
PROFILE_DIR = os.path.join(ROOT, "profiles")


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("hbm_gbs", FALLBACK_HBM_GBS), d.get("bf16_tflops", FALLBACK_BF16_TFLOPS), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def row_bytes(case) -> int:
    """Bytes of one cached row: W bf16 numbers, or an MX row (W codes of 1 byte for MXFP8, of
    half a byte for MXFP4, plus one scale byte per 32-element block)."""
    s = case["shape"]
    kv = case.get("kv", "")
    if kv == "mxfp8":
        return s.width + s.width // 32
    if kv == "mxfp4":
        return s.width // 2 + s.width // 32
    return s.width * 2


def workload_numbers(case, form=""):
    """Algorithmic bytes and FLOPs of one attention launch (the split-attention kernel).
    Decode: cache rows read once (L*row_bytes: L*W*2 for bf16), queries (n_h*W*2), outputs (n_h*(d_c*2+4)) per
    sequence; FLOPs 2*L*n_h*(W + d_c) per sequence (scores plus weighted sum).
    Causal prefill of T queries: the T cache rows once, T queries and outputs; query i
    attends i+1 tokens, so FLOPs 2*n_h*(W + d_c)*T(T+1)/2."""
    s = case["shape"]
    Wd = s.width
    per_q = s.n_heads * Wd * 2 + s.n_heads * (s.d_latent * 2 + 4)
    if "T" in case and form == "unabsorbed":
        # the flash kernel: query [T, n_h, d_h + d_r], K and V [T, n_h, d_h] and k_rope [T, d_r]
        # read once, o [T, n_h, d_h] and lse written; 2 n_h (d_h + d_r + d_h) FLOPs per
        # (query, visible key)
        T, H, dh, dr = int(case["T"]), s.n_heads, s.d_nope, s.d_rope
        bytes_ = T * H * (dh + dr) * 2 + 2 * T * H * dh * 2 + T * dr * 2 + T * H * (dh * 2 + 4)
        return bytes_, H * (dh + dr + dh) * T * (T + 1)
    if "T" in case:
        T = int(case["T"])
        return T * Wd * 2 + T * per_q, s.n_heads * (Wd + s.d_latent) * T * (T + 1)
    L = case["seq_lens"].astype(np.int64)
    bytes_ = int(np.sum(L * row_bytes(case) + per_q))
    flops = int(np.sum(2 * L * s.n_heads * (Wd + s.d_latent)))
    return bytes_, flops


# the sources each profiled kernel is compiled from (its own header and the headers it includes)
KERNEL_SOURCES = {
    "tc_attention": ["tc_attention.cuh", "tc_ptx.cuh", "sched.cuh", "mla_common.cuh", "simt_attention.cuh",
                     "mx_format.cuh"],
    "simt_attention": ["simt_attention.cuh", "sched.cuh", "mla_common.cuh", "mx_format.cuh"],
    "tc_gemm": ["tc_gemm.cuh", "tc_ptx.cuh", "mla_common.cuh", "mx_format.cuh"],
    "tc_flash": ["tc_flash.cuh", "tc_ptx.cuh", "mla_common.cuh"],
}


def code_text(src: str) -> str:
    """C++/CUDA source without its comments, trailing blanks and empty lines: what the
    compiler sees, so that an edit of a comment keeps a kernel's digest.  (String literals
    hold no comment markers in these sources; the inline PTX uses none.)"""
    out, i, n = [], 0, len(src)
    while i < n:
        if src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            j = min([k for k in (src.find("//", i), src.find("/*", i)) if k >= 0] or [n])
            out.append(src[i:j])
            i = j
    lines = [l.rstrip() for l in "".join(out).split("\n")]
    return "\n".join(l for l in lines if l)


def source_digest(kernel_key=None, read=None):
    """Digest of a kernel's sources (all of csrc/ when kernel_key is None), comments left out.
    `read(name)` returns a file's text (default: the working tree's)."""
    csrc = os.path.join(ROOT, "mla_latent_kv_79_b300", "csrc")
    read = read or (lambda f: open(os.path.join(csrc, f)).read())
    h = hashlib.sha256()
    for f in KERNEL_SOURCES.get(kernel_key) or sorted(os.listdir(csrc)):
        h.update(code_text(read(f)).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_key: str, workload: str):
    """DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) from the committed
    ncu summary profiles/<kernel>_<workload>.md, or None when it is missing or the kernel's
    sources changed since that capture (the summary records their digest)."""
    p = os.path.join(PROFILE_DIR, f"{kernel_key}_{workload}.md")
    if not os.path.exists(p):
        return None
    fields = {}
    for line in open(p):
        line = line.strip().lstrip("-").strip()
        if ":" in line:
            k, v = line.split(":", 1)
            fields[k.strip().strip("`")] = v.strip().strip("`")
    if (fields.get("source_digest", "").split() or [""])[0] != source_digest(kernel_key):
        return None
    try:
        return int(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def job_throughput(local_ms: float, local_units: int, device="cpu"):
    """Whole-job throughput over all ranks of the default process group (or this process
    alone): units summed over ranks divided by the slowest rank's time.
    Returns (units per second, max ms over ranks, total units)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(local_ms)], dtype=torch.float64, device=device)
    u = torch.tensor([int(local_units)], dtype=torch.int64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dist.all_reduce(u, op=dist.ReduceOp.SUM)
    ms, units = float(t.item()), int(u.item())
    return units / (ms * 1e-3), ms, units


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1])); mx.append(float(parts[2])); power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None}


# ------------------------------------------------------------------------------------ reference arm

def oracle_heads(case, budget_bytes: int = 4 << 30) -> int:
    """Heads the CPU oracle times at once (a power of two dividing n_h): it restores K and V of
    every head in float64, so long sequences would need tens of GB; the work is exactly linear
    in heads."""
    sh = case["shape"]
    per_head = 2 * int(np.max(case["seq_lens"])) * sh.d_nope * 8
    h = sh.n_heads
    while h > 1 and (h * per_head > budget_bytes or sh.n_heads % h):
        h //= 2
    return h


def cpu_oracle_sample(case, seqs, out_proj: bool = False, heads=None):
    """Time the float64 oracle (un-absorbed: restore K and V, softmax attention, W_UV folded
    in by V, and W_O when out_proj) on sequences `seqs` with the first `heads` heads (all by
    default); an append workload also runs the appended token's down-projection.  Returns
    seconds."""
    import oracle.mla_oracle as O
    s = case["shape"]
    h = s.n_heads if heads is None else heads
    sc = O.default_scale(s.d_nope, s.d_rope)
    f = lambda a: W.to_f64(a, case["dtype"])  # noqa: E731
    w_uk, w_uv = f(case["w_uk"][:, :h * s.d_nope]), f(case["w_uv"][:, :h * s.d_nope])
    w_o = f(case["w_o"][:h * s.d_nope]) if out_proj else None
    appending = "x" in case and "append_pos" in case
    if appending:
        w_dkv, w_kr = f(case["w_dkv"]), f(case["w_kr"])
    t0 = time.perf_counter()
    for b in seqs:
        if appending:
            O.latent_kv(f(case["x"][b:b + 1]), w_dkv, w_kr, case["append_pos"][b:b + 1], s.rope_base)
        L = int(case["seq_lens"][b])
        rows = oracle_rows(case, b, L)
        q_r = O.rope_rotate(f(case["q_rope"][b][:h]), case["pos"][b], s.rope_base)
        o = O.attention_unabsorbed(f(case["q_nope"][b][:h]), q_r, rows[:, :s.d_latent], rows[:, s.d_latent:],
                                   w_uk, w_uv, sc)[0]
        if out_proj:
            O.output_projection(o.reshape(1, -1), w_o)
    return time.perf_counter() - t0


def oracle_rows(case, b: int, L: int):
    """The oracle's float64 view of sequence b's first L cached rows (an MX cache through the
    oracle's MX decoder)."""
    import oracle.mla_oracle as O
    kv = case.get("kv", "")
    if not kv:
        return W.to_f64(W.gather_rows(case["pool"], case["page_table"][b], L), case["dtype"])
    codes = W.gather_rows(case["codes"], case["page_table"][b], L).astype(np.int64)
    sc = W.gather_rows(case["scales"], case["page_table"][b], L).astype(np.int64)
    if kv == "mxfp4":
        codes = O.mx_unpack_e2m1(codes)
    return O.mx_decode_rows(codes, sc, "e4m3" if kv == "mxfp8" else "e2m1")


def oracle_sample_text(case, n_seq: int, n_all: int, heads: int, per_step: bool = False) -> str:
    sh = case["shape"]
    lens = case["seq_lens"][:n_seq]
    toks = f"{int(lens[0])} cached tokens" if lens.min() == lens.max() else \
        f"{int(lens.min())}-{int(lens.max())} cached tokens"
    who = "one sequence per step" if per_step else f"{n_seq} of {n_all} sequences"
    hs = f"all {sh.n_heads} heads" if heads == sh.n_heads else \
        f"{heads} of {sh.n_heads} heads, time scaled by {sh.n_heads // heads} (the work is linear in heads)"
    return f"{who} ({hs}, {toks}), un-absorbed float64 oracle"


def cpu_baseline(case, out_proj: bool = False, budget_s: float = 10.0):
    """The oracle timed on the host cores over a bounded sample of the workload: whole
    sequences in order until about budget_s of oracle time, all heads unless the float64
    restore would not fit (then a head subset, scaled up linearly)."""
    sh = case["shape"]
    B = int(case["seq_lens"].shape[0])
    heads = oracle_heads(case)
    n_seq, t_cpu = 0, 0.0
    while n_seq < B and (n_seq == 0 or t_cpu < budget_s):
        t_cpu += cpu_oracle_sample(case, [n_seq], out_proj, heads)
        n_seq += 1
    t_cpu *= sh.n_heads / heads
    return {"value": n_seq / t_cpu, "unit": UNIT, "cores": cores(), "kind": "oracle",
            "sample": oracle_sample_text(case, n_seq, B, heads)}


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    if W.WORKLOADS[args.workload].mode not in ("decode", "append_decode"):
        print(json.dumps({"impl": "reference", "unavailable": "the oracle arm times the decode workloads only"}),
              flush=True)
        return 0
    case = W.make_workload(args.workload)
    heads = oracle_heads(case)
    for _ in range(max(0, args.warmup)):
        cpu_oracle_sample(case, [0], args.out_proj, heads)
    ts = [cpu_oracle_sample(case, [0], args.out_proj, heads) * (case["shape"].n_heads / heads)
          for _ in range(args.steps)]
    t = sum(ts)
    value = args.steps / t
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_of(args.workload, case, args.out_proj),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores(), "kind": "oracle",
                         "sample": oracle_sample_text(case, 1, 1, heads, per_step=True)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def config_of(name, case, out_proj=False):
    s = case["shape"]
    w = W.WORKLOADS[name]
    extra = {"step": {"decode": "absorb_q + decode + out",
                      "append_decode": "cache_append (one token per sequence) + absorb_q + decode + out",
                      "prefill": "cache_append (T tokens) + absorb_q + causal prefill + out"}[w.mode]
             + (" + out_proj (W_O)" if out_proj else "")}
    if w.form == "unabsorbed":
        extra["step"] = ("cache_append (T tokens) + un-absorbed causal prefill (gather, restore K and V, "
                         "192-wide causal attention)" + (" + out_proj (W_O)" if out_proj else ""))
    if "T" in case:
        extra["query_tokens"] = int(case["T"])
    return {"workload": name, "batch": int(case["seq_lens"].shape[0]), **extra,
            "seq_len": int(case["seq_lens"].max()), "n_heads": s.n_heads, "d_nope": s.d_nope,
            "d_rope": s.d_rope, "d_latent": s.d_latent, "page_size": s.page_size,
            "page_table": "shuffled", "cache": {"": "bf16 rows", "mxfp8": "MXFP8 (E4M3, 32-element E8M0 blocks)",
                                                 "mxfp4": "MXFP4 (E2M1, 32-element E8M0 blocks)"}[w.kv],
            "l2": "flushed between steps (256 MB write, then read back so no dirty lines remain)"}


def query_config(query: str) -> dict:
    if query == "given":
        return {}
    return {"query": {"direct": "x . W_Q, x . W_QR, then absorb_q (in the step)",
                      "compressed": "c_q = x . W_DQ, RoPE query c_q . W_QR, absorbed query from c_q with "
                                    "W_UQ folded into W_UK (in the step; d_cq = d_c)"}[query]}


# ------------------------------------------------------------------------------------ our arm

def run_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    from mla_latent_kv_79_b300 import build
    if rank == 0 or world == 1:
        build.build()
    if world > 1:
        dist.barrier()
    import mla_latent_kv_79_b300 as M

    case = W.make_workload(args.workload)
    mode = W.WORKLOADS[args.workload].mode
    if mode == "tiny_decode":
        raise SystemExit("the tiny fp32 workload is a parity case, not a benchmark")
    s = case["shape"]
    cfg = M.MLAConfig.from_shape(s, case["dtype"])
    dt = case["dtype"]
    dev = lambda a: W.to_device(a, dt)  # noqa: E731
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()  # noqa: E731
    if case.get("kv"):
        kvf = {"mxfp8": M.MLA_KV_MXFP8, "mxfp4": M.MLA_KV_MXFP4}[case["kv"]]
        cache = M.PagedCache(torch.from_numpy(case["codes"]).cuda(), i32(case["page_table"]),
                             i32(case["seq_lens"]), kvf, torch.from_numpy(case["scales"]).cuda())
    else:
        cache = M.PagedCache(dev(case["pool"]), i32(case["page_table"]), i32(case["seq_lens"]))
    q_nope, q_rope = dev(case["q_nope"]), dev(case["q_rope"])
    prefill = mode == "prefill"
    unabsorbed = W.WORKLOADS[args.workload].form == "unabsorbed"
    pos = i32(case["append_pos"] if prefill else case["pos"])
    w_uk, w_uv = dev(case["w_uk"]), dev(case["w_uv"])
    w_o = dev(case["w_o"]) if args.out_proj else None
    appending = mode in ("append_decode", "prefill")
    if appending:
        x, w_dkv, w_kr = dev(case["x"]), dev(case["w_dkv"]), dev(case["w_kr"])
        a_seq, a_pos = i32(case["append_seq"]), i32(case["append_pos"])
    B = int(case["T"]) if prefill else int(case["seq_lens"].shape[0])  # query tokens per step
    q_cat = torch.empty((B, s.n_heads, s.width), dtype=cfg.torch_dtype, device="cuda")
    o_lat = torch.empty((B, s.n_heads, s.d_latent), dtype=cfg.torch_dtype, device="cuda")
    lse = torch.empty((B, s.n_heads), dtype=torch.float32, device="cuda")
    o = torch.empty((B, s.n_heads * s.d_nope), dtype=cfg.torch_dtype, device="cuda")
    out = torch.empty((B, s.d_model), dtype=cfg.torch_dtype, device="cuda") if args.out_proj else None
    ws = M.alloc_workspace(cfg)
    if unabsorbed:
        import ctypes
        nb = ctypes.c_size_t(0)
        M.lib().mla_prefill_unabsorbed_workspace_size(ctypes.byref(cfg.c()), 0, B, ctypes.byref(nb))
        uws = torch.empty(int(nb.value), dtype=torch.uint8, device="cuda")
    # the query side of the step: given (q_nope, q_rope as inputs), direct (x . W_Q, x . W_QR) or
    # compressed (c_q = x . W_DQ, RoPE query c_q . W_QR, absorbed query with W_UQ folded into W_UK)
    if args.query != "given":
        qrng = np.random.default_rng(7 + B)
        xq = dev(W.quantise(W.normal(qrng, (B, s.d_model)), dt))
        if args.query == "direct":
            w_q = dev(W.weight(qrng, s.d_model, s.n_heads * s.d_nope, dt))
            w_qr = dev(W.weight(qrng, s.d_model, s.n_heads * s.d_rope, dt))
        else:
            d_cq = s.d_latent
            w_dq = dev(W.weight(qrng, s.d_model, d_cq, dt))
            w_qr = dev(W.weight(qrng, d_cq, s.n_heads * s.d_rope, dt))
            w_uqk = M.mla_fold_uq_uk(cfg, dev(W.weight(qrng, d_cq, s.n_heads * s.d_nope, dt)), w_uk)
            c_q = torch.empty((B, d_cq), dtype=cfg.torch_dtype, device="cuda")
        qn_buf = torch.empty_like(q_nope)
        qr_buf = torch.empty_like(q_rope)
        q_in = (xq,)
    else:
        q_in = (q_nope, q_rope)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    flush_words = flush.view(torch.int64)
    stream = torch.cuda.current_stream()

    def flush_l2():
        # evict the step's data from L2 with a 256 MB write, then read the buffer back, so that
        # the flush leaves clean lines behind and the timed step pays no write-back of the
        # flush's own data (measured on B300: a dirty 126 MB L2 slowed a 75 MB cold read by 20 %)
        flush.zero_()
        flush_words.sum()

    def step(qi=q_in, xx=None, oo=o, ll=lse, ff=out):
        if appending:  # the same positions every step: the cache ends each step identical
            M.mla_cache_append(cfg, cache, x if xx is None else xx, w_dkv, w_kr, a_seq, a_pos, stream=stream)
        if args.query == "direct":
            qn, qr = M.mla_query_proj(cfg, qi[0], w_q, w_qr, q_nope=qn_buf, q_rope=qr_buf, stream=stream)
        elif args.query == "compressed":
            M.mla_query_latent(cfg, qi[0], w_dq, c_q=c_q, stream=stream)
            M.mla_query_up(cfg, c_q, None, w_qr, q_rope=qr_buf, stream=stream)
            M.mla_absorb_q_compressed(cfg, c_q, qr_buf, pos, w_uqk, q_cat=q_cat, stream=stream)
        else:
            qn, qr = qi
        if unabsorbed:
            M.mla_prefill_unabsorbed(cfg, cache, 0, 0, qn, qr, w_uk, w_uv, o=oo, lse=ll, workspace=uws, stream=stream)
            if args.out_proj:
                M.mla_out_proj(cfg, oo, w_o, out=ff, stream=stream)
            return
        if args.query != "compressed":
            M.mla_absorb_q(cfg, qn, qr, pos, w_uk, q_cat=q_cat, stream=stream)
        if prefill:
            M.mla_prefill(cfg, cache, 0, 0, q_cat, o_lat=o_lat, lse=ll, workspace=ws, stream=stream)
        else:
            M.mla_decode(cfg, cache, q_cat, o_lat=o_lat, lse=ll, workspace=ws, stream=stream)
        M.mla_out(cfg, o_lat, w_uv, o=oo, stream=stream)
        if args.out_proj:  # the layer output, out = o . W_O
            M.mla_out_proj(cfg, oo, w_o, out=ff, stream=stream)

    warm = max(3, args.warmup)
    clocks = ClockSampler(local)
    clocks.start()
    for _ in range(warm):
        flush_l2()
        step()
    torch.cuda.synchronize()
    assert M.mla_get_device_error() == 0

    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for a, b in kev:  # create the events so their handles exist
        a.record(); b.record()
    torch.cuda.synchronize()
    lib = M.lib()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = lib.mla_kernel_launches()
    for i in range(K):
        flush_l2()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    launches = lib.mla_kernel_launches() - launches0
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    # the attention kernel's own duration, from events the library records around its launch
    # on the same stream; a separate pass, because events between two kernels keep the second
    # from starting early (programmatic dependent launch) and would slow the timed steps
    for i in range(K):
        flush_l2()
        lib.mla_set_attention_events(kev[i][0].cuda_event, kev[i][1].cuda_event)
        step()
    lib.mla_set_attention_events(None, None)
    torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    kern_ms = [a.elapsed_time(b) for a, b in kev]
    value, total_ms, tokens_total = job_throughput(sum(step_ms), B * K, "cuda")
    path = M.mla_last_attention_path()
    assert M.mla_get_device_error() == 0

    # end to end through host buffers: per step, the step's inputs come in from pinned host
    # memory in one copy and its results go back in one copy (the device tensors the path reads
    # and writes are views of one staging buffer each way, as a serving loop would pack them)
    def staging(tensors, pinned):
        offs, n = [], 0
        for t in tensors:
            offs.append(n)
            n += (t.numel() * t.element_size() + 15) // 16 * 16
        buf = torch.empty(n, dtype=torch.uint8, device="cpu" if pinned else "cuda")
        if pinned:
            buf = buf.pin_memory()
        views = [buf[o_:o_ + t.numel() * t.element_size()].view(t.dtype).view(t.shape) for o_, t in zip(offs, tensors)]
        return buf, views
    ins = list(q_in) + ([x] if appending else [])
    d_in, e_in = staging(ins, pinned=False)
    h_in, h_in_views = staging(ins, pinned=True)
    for hv, t in zip(h_in_views, ins):
        hv.copy_(t)
    results = [out, lse] if args.out_proj else [o, lse]
    d_out, e_res = staging(results, pinned=False)
    h_out, _ = staging(results, pinned=True)
    if args.out_proj:
        e_o, e_lse, e_f = o, e_res[1], e_res[0]
    else:
        e_o, e_lse, e_f = e_res[0], e_res[1], out
    eev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    for i in range(K):
        flush_l2()
        eev[i][0].record(stream)
        d_in.copy_(h_in, non_blocking=True)
        nq = len(q_in)
        step(tuple(e_in[:nq]), e_in[nq] if appending else None, e_o, e_lse, e_f)
        h_out.copy_(d_out, non_blocking=True)
        eev[i][1].record(stream)
    torch.cuda.synchronize()
    clock = clocks.stop()
    e2e_value, e2e_ms, _ = job_throughput(sum(a.elapsed_time(b) for a, b in eev), B * K, "cuda")
    if world > 1:
        dist.barrier()

    if rank != 0:
        dist.destroy_process_group()
        return 0

    alg_bytes, alg_flops = workload_numbers(case, W.WORKLOADS[args.workload].form)
    hbm, tflops, src = peaks()
    k_mean_s = (sum(kern_ms) / K) * 1e-3
    achieved = alg_bytes / k_mean_s / 1e9
    tensor_bound = alg_flops / (tflops * 1e12) > alg_bytes / (hbm * 1e9)
    kernel_key = {2: "tc_attention", 3: "tc_flash"}.get(path, "simt_attention")
    line = {
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": K,
        "warmup": warm,
        "ms_per_step": total_ms / K,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {**config_of(args.workload, case, args.out_proj), **query_config(args.query)},
        "roofline": {"bound": "tensor" if tensor_bound else "hbm",
                     "achieved": alg_flops / k_mean_s / 1e12 if tensor_bound else achieved,
                     "peak": tflops if tensor_bound else hbm, "unit": "TFLOP/s" if tensor_bound else "GB/s",
                     "frac": (alg_flops / k_mean_s / 1e12 / tflops) if tensor_bound else achieved / hbm,
                     "traffic": ncu_traffic(kernel_key, args.workload), "gbs": achieved,
                     "kernel": kernel_key, "kernel_us": k_mean_s * 1e6,
                     "algorithmic_bytes": alg_bytes, "algorithmic_flops": alg_flops,
                     "tflops": alg_flops / k_mean_s / 1e12, "peak_source": src,
                     "tensor_frac": alg_flops / k_mean_s / 1e12 / tflops,
                     "roofline_us": 1e6 * max(alg_bytes / (hbm * 1e9), alg_flops / (tflops * 1e12))},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": int(h_in.numel()),
                "d2h_bytes_per_step": int(h_out.numel())},
        "gpu_launches": int(launches),
        "clocks": clock,
        "cpu_baseline": None,
        "step_us_median": 1e3 * statistics.median(step_ms),
    }
    if not args.no_cpu_baseline and not prefill:
        line["cpu_baseline"] = cpu_baseline(case, args.out_proj)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode_b16_l4096", choices=sorted(W.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--query", default="given", choices=["given", "direct", "compressed"],
                    help="query side in the step: given q_nope/q_rope, or from x (direct or compressed)")
    ap.add_argument("--out-proj", action="store_true",
                    help="add the output projection over the heads (W_O) to the timed step")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
