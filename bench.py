#!/usr/bin/env python3
"""Decode-step benchmark: one JSON line.

A step is one pass of the whole decode hot path over one batch: kv_append_rope
(RoPE + append of the new token) and gqa_decode_attention (attention over the
cache, plus the split combine when it splits), all through the C ABI.
The default workload is the Llama-style GQA decode step (batch 32, 32 query
heads, 8 KV heads, head_dim 128, 4096-token bf16 cache, RoPE base 10000).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--cache native|u8|fp8] [--window W]

``value`` is the achieved HBM throughput of the step in GB/s (algorithmic
bytes / device time, summed over ranks); ``ms_per_step`` gives the step time.
Under torchrun each rank runs its own batch (weak scaling, no collective on
the data path). ``--impl reference`` times the fp64 CPU oracle on the host
cores instead, one (sequence, kv head) unit of the same workload per step.
``--cache u8`` runs the same workload over a uint8 cache (codes plus a float32
(scale, zero point) pair per cached row, as the pages' QuantizedKVCache);
``--cache fp8`` over an fp8 e5m2 cache (one byte per element, no scale).
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

# The oracle legs run single-threaded: pin BLAS before numpy loads.
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from synthetic import make_contiguous_case, make_e5m2_cache, make_paged_case, make_u8_cache, normal, workload  # noqa: E402

METRIC = "decode-attention HBM GB/s (fraction of GB300 peak) and µs/step at 1 GPU"
UNIT = "GB/s"
DEFAULT_WORKLOAD = "gqa4k"
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ["decode_mma.cu", "decode_mma_paged.cu", "decode_mma_u8.cu", "attn_tc05.cu", "attn_tc05_keys.cu",
                  "attn_tc05_widen.cu",
                  "mma_warp.cuh", "tc05.cuh", "quant.cuh",
                  "rope.cuh", "ptx.cuh", "launch.h"]


# ------------------------------------------------------------------ helpers
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, world: int) -> float:
    """Largest value of x over all ranks (the slowest rank's time)."""
    if world <= 1:
        return x
    import torch.distributed as dist

    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def throughput_gbs(world: int, bytes_per_step: int, ms_per_step: float) -> float:
    """Whole-job GB/s: every rank streams its own batch's bytes each step."""
    return world * bytes_per_step / (ms_per_step * 1e-3) / 1e9


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, STREAM-style copy)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, earlier GB300 measurement)"


def kernel_source_hash():
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "mqa_decode_attention_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload_name: str):
    """DRAM bytes per decode launch from the committed ncu summary, if it was
    taken on the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        e = d.get(workload_name)
        if e and e.get("source_sha") == kernel_source_hash():
            return float(e["dram_bytes_per_launch"])
    except (OSError, ValueError, KeyError):
        pass
    return None


def attended(lens, window: int, n_new: int = 1):
    """Tokens each sequence's queries read: all L, or with a window the last
    `window` tokens of each of its n_new queries (their union)."""
    return lens.clamp(max=window + n_new - 1) if window > 0 else lens


def row_bytes(w, cache: str) -> int:
    """Bytes of one cached (token, kv head) row of K (or V): head_dim values,
    or head_dim uint8 codes plus the float32 (scale, zero point) pair."""
    if cache == "u8":
        return w.head_dim + 8
    return w.head_dim if cache == "fp8" else w.head_dim * w.esize


def step_bytes(w, lens, out_esize, window: int = 0, cache: str = "native", n_new: int = 1):
    """Algorithmic bytes of one step: every attended K/V byte read once
    (including the new tokens; once for all n_new queries of a sequence),
    q_new read, out written, k_new/v_new read and their slots written, and
    (paged) the block-table entries used."""
    es = w.esize  # q_new / k_new / v_new
    att = attended(lens, window, n_new)
    kv = 2 * int(att.sum()) * w.h_kv * row_bytes(w, cache)
    q = n_new * w.batch * w.h_q * w.head_dim * es
    out = n_new * w.batch * w.h_q * w.head_dim * out_esize
    append = 2 * n_new * w.batch * w.h_kv * (w.head_dim * es + row_bytes(w, cache))
    table = 4 * int(((att + w.page_size - 1) // w.page_size).sum()) if w.paged else 0
    return kv + q + out + append + table


def attention_bytes(w, lens, out_esize, window: int = 0, cache: str = "native", n_new: int = 1):
    """Algorithmic bytes of one gqa_decode_attention launch: K/V of every
    attended token, q_rot (fp32) read, out written, block-table entries (paged)."""
    lens = attended(lens, window, n_new)
    kv = 2 * int(lens.sum()) * w.h_kv * row_bytes(w, cache)
    q = n_new * w.batch * w.h_q * w.head_dim * 4
    out = n_new * w.batch * w.h_q * w.head_dim * out_esize
    table = 4 * int(((lens + w.page_size - 1) // w.page_size).sum()) if w.paged else 0
    return kv + q + out + table


class ClockSampler:
    """nvidia-smi clocks / throttle reasons, sampled every 100 ms in a thread."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: str):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", gpu_index, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.monotonic(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        sel = [p for t, p in self.samples if t0 <= t <= t1]
        if not sel:
            sel = [p for _, p in self.samples[-5:]]
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(p[1]) for p in sel if num(p[1]) is not None]
        mx = [num(p[2]) for p in sel if num(p[2]) is not None]
        pw = [num(p[3]) for p in sel if num(p[3]) is not None]
        reasons = sorted({name for p in sel for name, v in zip(self.NAMES, p[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(sel), "power_w_max": max(pw) if pw else None}


def gpu_index_for(local_rank: int) -> str:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [x.strip() for x in vis.split(",") if x.strip()]
        if local_rank < len(ids):
            return ids[local_rank]
    return str(local_rank)


# ----------------------------------------------------------- inputs / oracle
U8_SEED = 77


S_QM, S_KM, S_VM = 21, 22, 23  # seeded streams of multi-token q, k, v


def build_case(w, device, cache: str = "native", n_new: int = 1):
    """The workload's seeded inputs. With cache "u8" the K/V caches are
    replaced by uint8 codes and (scale, zero point) pairs of the same rows
    (attributes u8 = synthetic.U8Cache), with cache "fp8" by fp8 e5m2 caches
    (attribute f8 = (K, V)). With n_new > 1 the new tokens are [B, n_new, H, d]
    and pos = seq_lens - n_new."""
    case = make_paged_case(w, device) if w.paged else make_contiguous_case(w, device)
    case.u8 = None
    case.f8 = None
    case.n_new = n_new
    if n_new > 1:
        case.q_new = normal((w.batch, n_new, w.h_q, w.head_dim), w.seed, S_QM, w.dtype, device)
        case.k_new = normal((w.batch, n_new, w.h_kv, w.head_dim), w.seed, S_KM, w.dtype, device)
        case.v_new = normal((w.batch, n_new, w.h_kv, w.head_dim), w.seed, S_VM, w.dtype, device)
        case.pos = (case.seq_lens - n_new).to(torch.int32)
    if cache in ("u8", "fp8"):
        if w.paged:
            rows = (case.num_pages, w.h_kv, case.page_size)
            case.k_pool = case.v_pool = None
        else:
            rows = (w.batch, w.h_kv, case.capacity)
            case.k_cache = case.v_cache = None
        if cache == "u8":
            case.u8 = make_u8_cache(rows, w.head_dim, U8_SEED, device=device)
        else:
            case.f8 = make_e5m2_cache(rows, w.head_dim, U8_SEED, device=device)
    return case


def _rows(w, case, cache_t, b, j, L):
    """Rows [0, L) of kv head j of sequence b from a cache tensor."""
    if w.paged:
        n = (L + w.page_size - 1) // w.page_size
        pages = case.block_table[b, :n].long()
        return cache_t[pages, j].reshape(-1, *cache_t.shape[3:])[:L].cpu()
    return cache_t[b, j, :L].cpu()


def unit_inputs(w, case, units):
    """CPU copies of the inputs of (b, j) units, taken before any step runs."""
    G = w.group
    out = []
    lens = case.seq_lens.cpu()
    for b, j in units:
        L = int(lens[b])
        if case.n_new > 1:  # [n, G, d] queries, [n, d] k / v of the unit
            u = dict(b=b, j=j, L=L, q=case.q_new[b, :, j * G:(j + 1) * G].cpu(), k=case.k_new[b, :, j].cpu(),
                     v=case.v_new[b, :, j].cpu(), n=case.n_new)
        else:
            u = dict(b=b, j=j, L=L, q=case.q_new[b, j * G:(j + 1) * G].cpu(), k=case.k_new[b, j].cpu(),
                     v=case.v_new[b, j].cpu(), n=1)
        if case.u8 is not None:
            c = case.u8
            u.update(Kc=_rows(w, case, c.k_codes, b, j, L), Ks=_rows(w, case, c.k_sz, b, j, L),
                     Vc=_rows(w, case, c.v_codes, b, j, L), Vs=_rows(w, case, c.v_sz, b, j, L))
        elif case.f8 is not None:
            u.update(K8=_rows(w, case, case.f8[0].view(torch.uint8), b, j, L),
                     V8=_rows(w, case, case.f8[1].view(torch.uint8), b, j, L))
        else:
            kc, vc = (case.k_pool, case.v_pool) if w.paged else (case.k_cache, case.v_cache)
            u.update(K=_rows(w, case, kc, b, j, L), V=_rows(w, case, vc, b, j, L))
        out.append(u)
    return out


def numpy_units(w, units, out_esize, cache: str, n_new: int, window: int):
    """The units as numpy arrays for oracle.cores: bf16 values as their 16-bit
    patterns (fp32 values as float32), byte caches as stored, and each unit's
    algorithmic bytes."""
    import numpy as np

    span = (window + n_new - 1) if window else 1 << 30
    out = []
    for u in units:
        v = {"L": np.array(u["L"]), "n": np.array(u["n"]),
             "bytes": np.array(unit_bytes(w, min(u["L"], span), out_esize, cache, n_new))}
        for key, t in u.items():
            if not isinstance(t, torch.Tensor):
                continue
            if t.dtype == torch.bfloat16:
                v[key] = t.contiguous().view(torch.int16).numpy().view(np.uint16)
            elif t.dtype == torch.float32:
                v[key] = t.numpy()
            else:
                v[key] = t.numpy()
        out.append(v)
    return out


def oracle_meta(w, window: int) -> dict:
    return {"scale": 1.0 / math.sqrt(w.head_dim), "rope_base": w.rope_base, "window": window, "dtype": w.dtype,
            "bf16_bits": w.dtype == "bf16"}


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_baseline(w, units, out_esize, cache: str, n_new: int, window: int, seconds: float, runs: int = 3):
    """The oracle's decode step timed on the host cores over a sample of units:
    single-threaded in this process and on every core (one process per core,
    oracle.cores), each the median of `runs` runs of about `seconds` seconds.
    Returns (single, all_cores, outputs of the distinct units)."""
    import subprocess
    import tempfile

    from oracle import cores  # test infrastructure: the CPU-baseline leg only

    nu = numpy_units(w, units, out_esize, cache, n_new, window)
    meta = oracle_meta(w, window)
    with tempfile.TemporaryDirectory() as tmp:
        path = os.path.join(tmp, "units.npz")
        cores.save_units(path, nu, meta)
        loaded, _ = cores.load_units(path)
        outs = [cores.run_unit(u, meta) for u in loaded]  # also the warm-up
        single = []
        for _ in range(runs):
            nb, nd, secs = cores.run_for(loaded, meta, seconds)
            single.append({"bytes": nb, "units": nd, "wall_s": secs})
        del loaded
        procs = host_cores()
        r = subprocess.run([sys.executable, "-m", "oracle.cores", path, "--seconds", str(seconds), "--runs",
                            str(runs), "--procs", str(procs)], cwd=ROOT, capture_output=True, text=True,
                           timeout=600)
        if r.returncode != 0:
            raise RuntimeError("oracle.cores failed: " + r.stderr[-2000:])
        multi = json.loads(r.stdout.strip().splitlines()[-1])

    def med(rs):
        rates = sorted(x["bytes"] / x["wall_s"] / 1e9 for x in rs)
        return rates[len(rates) // 2], rates

    s_med, s_all = med(single)
    m_med, m_all = med(multi["runs"])
    return ({"value": s_med, "runs_gbs": s_all, "cores": 1, "seconds_per_run": seconds},
            {"value": m_med, "runs_gbs": m_all, "cores": multi["procs"], "seconds_per_run": seconds}, outs)


def unit_bytes(w, L, out_esize, cache: str = "native", n_new: int = 1):
    es = w.esize
    return (2 * L * row_bytes(w, cache) + n_new * w.group * w.head_dim * (es + out_esize)
            + 2 * n_new * (w.head_dim * es + row_bytes(w, cache)))


# ------------------------------------------------ every workload, L2-controlled
SWEEP = ["gqa4k", "mqa8k", "paged", "long"]


def percentiles(xs):
    xs = sorted(xs)
    q = statistics.quantiles(xs, n=10, method="inclusive")
    return {"median": round(statistics.median(xs), 6), "p10": round(q[0], 6), "p90": round(q[-1], 6)}


def layout_for(m, w, case, window: int = 0):
    if w.paged:
        return m.layout_paged(case.k_pool, case.v_pool, case.block_table, w.h_q, window=window)
    return m.layout_contiguous(case.k_cache, case.v_cache, w.h_q, window=window)


def measure_workload(m, name, dev, stream, n_timed, n_warm, flush, sampler, l2_bytes, peak):
    """One workload's decode step (mqa_decode_step: RoPE, append, attention,
    the combine when it splits) at its own split count, two ways:
    isolated -- each step preceded by an L2 flush (a read of a buffer twice
    the L2 size), CUDA events around the step alone: median, p10, p90;
    back to back -- steps one after another over enough identical copies of
    the cache that at least 4x the L2 size streams between two reads of the
    same copy. Returns the entry for the bench line."""
    w = workload(name)
    lens = None
    copies = []
    one = None
    while True:
        case = build_case(w, dev)
        lay = layout_for(m, w, case)
        lens = case.seq_lens.cpu()
        max_len = int(lens.max())
        bufs = m.DecodeBuffers.allocate(lay, max_len, num_splits=w.num_splits, device=dev)
        copies.append((case, lay, bufs))
        if one is None:
            one = step_bytes(w, lens, bufs.out.element_size())
        if len(copies) * one >= 4 * l2_bytes:
            break
    scale = 1.0 / math.sqrt(w.head_dim)
    splits = w.num_splits if w.num_splits > 0 else m.choose_splits(copies[0][1], max_len, 0, 1)

    def step(i):
        case, lay, bufs = copies[i % len(copies)]
        m.decode_step(lay, case.q_new, case.k_new, case.v_new, case.pos, case.seq_lens, max_len, bufs, w.rope_base,
                      scale, w.num_splits, 0, stream)

    for i in range(n_warm):
        step(i)
    torch.cuda.synchronize()
    t0 = time.monotonic()
    e0 = [torch.cuda.Event(enable_timing=True) for _ in range(n_timed)]
    e1 = [torch.cuda.Event(enable_timing=True) for _ in range(n_timed)]
    for i in range(n_timed):
        flush()
        e0[i].record(stream)
        step(i)
        e1[i].record(stream)
    torch.cuda.synchronize()
    iso = [e0[i].elapsed_time(e1[i]) for i in range(n_timed)]
    # back to back for at least half a second, so that the clock sampler sees this workload
    n_b2b = max(n_timed, int(0.5e3 / statistics.median(iso)))
    b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    b0.record(stream)
    for i in range(n_b2b):
        step(i)
    b1.record(stream)
    torch.cuda.synchronize()
    t1 = time.monotonic()
    b2b = b0.elapsed_time(b1) / n_b2b
    for _, _, bufs in copies:
        err = int(bufs.err.item())
        if err != 0:
            raise RuntimeError(f"{name}: device error word {err:#x}")
    pc = percentiles(iso)
    gbs = one / (pc["median"] * 1e-3) / 1e9
    traffic = ncu_traffic(name)
    entry = {
        "shape": (f"batch {w.batch}, H_q {w.h_q}, H_kv {w.h_kv}, head_dim {w.head_dim}, "
                  + (f"{w.page_size}-token pages, lengths U[{w.len_lo},{w.len_hi}]" if w.paged
                     else f"{w.seq_len} tokens/seq")),
        "num_splits": splits,
        "bytes_per_step": one,
        "ms_per_step": pc,
        "gbs": round(gbs, 2),
        "frac_of_measured": round(gbs / peak, 4),
        "frac_of_8000": round(gbs / 8000.0, 4),
        "back_to_back": {"ms_per_step": round(b2b, 6), "gbs": round(one / (b2b * 1e-3) / 1e9, 2),
                         "frac_of_measured": round(one / (b2b * 1e-3) / 1e9 / peak, 4),
                         "cache_copies": len(copies), "steps": n_b2b},
        "ncu_traffic_ratio": round(traffic / one, 4) if traffic else None,
        "steps": n_timed,
        "clocks": sampler.summary(t0, t1),
        "l2": (f"isolated: L2 flushed before each step (read of {2 * l2_bytes / 1e6:.0f} MB); back to back: "
               f"{len(copies)} cache cop{'y' if len(copies) == 1 else 'ies'}, {len(copies) * one / 1e6:.0f} MB "
               f"streamed between reads of a copy ({l2_bytes / 1e6:.0f} MB L2)"),
    }
    del copies
    torch.cuda.empty_cache()
    return entry


def measure_workloads(m, dev, stream, n_timed, sampler, peak):
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or (129 << 20))
    flush_buf = torch.ones(2 * l2 // 4, dtype=torch.float32, device=dev)

    def flush():
        flush_buf.sum()

    out = {}
    for name in SWEEP:
        out[name] = measure_workload(m, name, dev, stream, n_timed, 10, flush, sampler, l2, peak)
    del flush_buf
    torch.cuda.empty_cache()
    return out


def tiny_parity(m, dev):
    """The tiny workload (fp32, batch 1, 4 / 2 heads, head_dim 64, a 5-token
    prompt then decoding until 16 attention evaluations) token by token
    through the library, against the oracle's cached sequence."""
    import numpy as np

    import oracle  # test infrastructure: the CPU-baseline leg only
    from synthetic import make_tiny_sequence

    w = workload("tiny")
    seq = make_tiny_sequence(w)
    scale = 1.0 / math.sqrt(w.head_dim)
    n = seq.prompt_len + seq.decode_evals - 1
    ref, _, _, _ = oracle.run_cached_sequence(seq.q, seq.k, seq.v, seq.prompt_len, seq.decode_evals, w.rope_base,
                                              scale, "f32")
    kc = torch.zeros(w.batch, w.h_kv, n, w.head_dim, dtype=torch.float32, device=dev)
    vc = torch.zeros_like(kc)
    lay = m.layout_contiguous(kc, vc, w.h_q)
    bufs = m.DecodeBuffers.allocate(lay, n, num_splits=1, variant=1, device=dev)
    outs = []
    for p in range(n):
        lens = torch.full((w.batch,), p + 1, dtype=torch.int32, device=dev)
        m.decode_step(lay, seq.q[p].to(dev), seq.k[p].to(dev), seq.v[p].to(dev), lens - 1, lens, p + 1, bufs,
                      w.rope_base, scale, num_splits=1, variant=1)
        if p >= seq.prompt_len - 1:
            outs.append(bufs.out.double().cpu().numpy())
    torch.cuda.synchronize()
    if int(bufs.err.item()) != 0:
        raise RuntimeError("tiny: device error word")
    err = float(np.max(np.abs(np.stack(outs) - ref)))
    return {"shape": "batch 1, H_q 4, H_kv 2, head_dim 64, fp32, prompt 5 then 16 attention evaluations",
            "max_abs_err": err, "tolerance": 1e-4, "path": "CUDA-core kernel, fp32 cache and output"}


# --------------------------------------------------------------- our arm
def bench_ours(args):
    import mqa_decode_attention_gb300 as m
    import numpy as np

    world, rank, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)

    w = workload(args.workload)
    if args.splits is not None:
        w = w.with_(num_splits=args.splits)
    if args.batch:
        w = w.with_(batch=args.batch)
    u8 = args.cache == "u8"
    f8 = args.cache == "fp8"
    byte = u8 or f8  # a one-byte cache: the uint8 / e5m2 kernels
    nn = args.n_new
    case = build_case(w, dev, args.cache, nn)
    lens_cpu = case.seq_lens.cpu()
    max_len = int(lens_cpu.max())
    if u8:
        c = case.u8
        if w.paged:
            lay = m.layout_paged(c.k_codes, c.v_codes, case.block_table, w.h_q, window=args.window,
                                 k_scale_zero=c.k_sz, v_scale_zero=c.v_sz)
        else:
            lay = m.layout_contiguous(c.k_codes, c.v_codes, w.h_q, window=args.window, k_scale_zero=c.k_sz,
                                      v_scale_zero=c.v_sz)
    elif f8:
        if w.paged:
            lay = m.layout_paged(case.f8[0], case.f8[1], case.block_table, w.h_q, window=args.window)
        else:
            lay = m.layout_contiguous(case.f8[0], case.f8[1], w.h_q, window=args.window)
    elif w.paged:
        lay = m.layout_paged(case.k_pool, case.v_pool, case.block_table, w.h_q, window=args.window)
    else:
        lay = m.layout_contiguous(case.k_cache, case.v_cache, w.h_q, window=args.window)
    variant = args.variant
    bufs = m.DecodeBuffers.allocate(lay, max_len, num_splits=w.num_splits, variant=variant, device=dev, n_new=nn)
    scale = 1.0 / math.sqrt(w.head_dim)
    splits_used = w.num_splits if w.num_splits > 0 else m.choose_splits(lay, max_len, variant, nn)
    out_es = bufs.out.element_size()
    sbytes = step_bytes(w, lens_cpu, out_es, args.window, args.cache, nn)
    abytes = attention_bytes(w, lens_cpu, out_es, args.window, args.cache, nn)
    stream = torch.cuda.current_stream()

    # CPU-baseline units (rank 0, N = 1), copied before any step touches the cache
    do_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    units = []
    if do_cpu:
        g = torch.Generator().manual_seed(w.seed)
        perm = torch.randperm(w.batch * w.h_kv, generator=g).tolist()
        n_units = args.cpu_units or min(len(perm), max(2 * host_cores(), 16))
        units = unit_inputs(w, case, [(u // w.h_kv, u % w.h_kv) for u in perm[:n_units]])

    def append():
        m.kv_append_rope_multi(lay, nn, case.q_new, case.k_new, case.v_new, case.pos, w.rope_base, bufs.q_rot,
                               bufs.err, stream)

    def attend():
        m.gqa_decode_attention_multi(lay, nn, bufs.q_rot, case.seq_lens, max_len, scale, w.num_splits, bufs.out,
                                     bufs.lse, bufs.workspace, variant, bufs.err, stream)

    def step_on(st):
        if nn > 1:
            m.decode_step_multi(lay, nn, case.q_new, case.k_new, case.v_new, case.pos, case.seq_lens, max_len, bufs,
                                w.rope_base, scale, w.num_splits, variant, st)
        else:
            m.decode_step(lay, case.q_new, case.k_new, case.v_new, case.pos, case.seq_lens, max_len, bufs,
                          w.rope_base, scale, w.num_splits, variant, st)

    def step():
        step_on(stream)

    # the library's routing, as it reports it: the launches of one step and
    # whether the append runs inside the attention launch; a split step with
    # one launch fewer than append + attention + combine merged its splits
    # inside the attention launch
    launches_per_step, fused = m.step_launches(lay, max_len, w.num_splits, variant, nn)
    assert launches_per_step > 0, "the library refuses this step"
    merged = splits_used > 1 and launches_per_step == (1 if fused else 2)
    # 32 or more query rows per kv head (G x n_new) with head_dim 128 run on the
    # tcgen05 kernel: contiguous bf16, paged bf16 with several tokens,
    # contiguous e5m2 with several tokens
    tc05 = (variant in (0, 2) and w.head_dim == 128 and w.group * nn >= 32
            and ((w.dtype == "bf16" and not byte and (not w.paged or nn > 1))
                 or (args.cache == "fp8" and not w.paged and nn > 1)))

    # warm-up (at least W steps and at least ~1 s, so the clock sampler sees load)
    sampler = ClockSampler(gpu_index_for(local))
    t_warm = time.monotonic()
    n_warm = 0
    while n_warm < args.warmup or time.monotonic() - t_warm < args.warm_seconds:
        step()
        n_warm += 1
        if n_warm % 256 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    t_clock0 = time.monotonic() - 0.5

    # timed region: K steps through mqa_decode_step, events at both ends
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    K = args.steps
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for _ in range(K):
        step()
    t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t_clock1 = time.monotonic()
    total_ms = t_start.elapsed_time(t_end)

    # per-launch durations: K more steps, an event on each side of every call.
    # When the step is a single launch (tensor cores, no split) this is that
    # kernel's own duration; with a split it also holds the combine.
    ev_s = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev_e = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for i in range(K):
        ev_s[i].record(stream)
        step()
        ev_e[i].record(stream)
    torch.cuda.synchronize()
    step_call_ms = statistics.fmean(ev_s[i].elapsed_time(ev_e[i]) for i in range(K))
    # the standalone calls, for reference (not part of the step)
    n_alone = min(K, 500)
    ea = [torch.cuda.Event(enable_timing=True) for _ in range(3 * n_alone)]
    for i in range(n_alone):
        ea[3 * i].record(stream)
        append()
        ea[3 * i + 1].record(stream)
        attend()
        ea[3 * i + 2].record(stream)
    torch.cuda.synchronize()
    append_ms = statistics.fmean(ea[3 * i].elapsed_time(ea[3 * i + 1]) for i in range(n_alone))
    attn_ms = statistics.fmean(ea[3 * i + 1].elapsed_time(ea[3 * i + 2]) for i in range(n_alone))
    err_word = int(bufs.err.item())
    if err_word != 0:
        raise RuntimeError(f"device error word {err_word:#x} after the timed steps")

    ms_per_step = max_over_ranks(total_ms, world) / K
    value = throughput_gbs(world, sbytes, ms_per_step)

    # end to end: the step's inputs (q, k, v, positions, lengths) packed in one
    # pinned host block and copied in with one host-to-device copy, the output
    # copied out, every step; the step reads views of a device block. As a
    # serving loop would, the copies run on their own streams: step k + 1's
    # inputs go in (double-buffered device block) while step k runs, and step
    # k's output comes out (double-buffered output) while step k + 1 runs.
    srcs = [case.q_new, case.k_new, case.v_new, case.pos, case.seq_lens]
    offs, h2d = [], 0
    for x in srcs:
        offs.append(h2d)
        h2d += (x.numel() * x.element_size() + 255) // 256 * 256
    host_blk = torch.empty(h2d, dtype=torch.uint8).pin_memory()
    for x, o in zip(srcs, offs):
        nb = x.numel() * x.element_size()
        host_blk[o:o + nb].copy_(x.detach().cpu().contiguous().view(-1).view(torch.uint8))
    dev_blks = [torch.empty(h2d, dtype=torch.uint8, device=dev) for _ in range(2)]
    view_sets = [[blk[o:o + x.numel() * x.element_size()].view(x.dtype).view(x.shape) for x, o in zip(srcs, offs)]
                 for blk in dev_blks]
    outs = [bufs.out, torch.empty_like(bufs.out)]
    host_outs = [torch.empty(bufs.out.shape, dtype=bufs.out.dtype).pin_memory() for _ in range(2)]
    d2h = host_outs[0].numel() * host_outs[0].element_size()
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of the block landed
    ev_step = [torch.cuda.Event() for _ in range(2)]  # the step that read the block / wrote the output is done
    ev_out = [torch.cuda.Event() for _ in range(2)]   # the output was copied out

    def e2e_step(k, st, first=False):
        a = k % 2
        if not first:
            s_in.wait_event(ev_step[a])  # step k - 2 read this block
        with torch.cuda.stream(s_in):
            dev_blks[a].copy_(host_blk, non_blocking=True)
        ev_in[a].record(s_in)
        st.wait_event(ev_in[a])
        if not first:
            st.wait_event(ev_out[a])  # step k - 2's output has left this buffer
        case.q_new, case.k_new, case.v_new, case.pos, case.seq_lens = view_sets[a]
        bufs.out = outs[a]
        step_on(st)
        ev_step[a].record(st)
        s_out.wait_event(ev_step[a])
        with torch.cuda.stream(s_out):
            host_outs[a].copy_(outs[a], non_blocking=True)
        ev_out[a].record(s_out)

    for k in range(4):
        e2e_step(k, stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    for k in range(K):
        e2e_step(k, stream)
    stream.wait_event(ev_out[(K - 1) % 2])
    stream.wait_event(ev_out[K % 2])
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_eager_ms = max_over_ranks(e0.elapsed_time(e1), world)

    # The same loop as a serving process runs it: E2E_GRAPH steps (copies in,
    # steps, copies out, their streams and events) captured once into a CUDA
    # graph and replayed; consecutive replays are serialised, so one copy in
    # and one copy out per replay are not overlapped
    E2E_GRAPH = 32
    reps = max(1, K // E2E_GRAPH)
    cap = torch.cuda.Stream(device=dev)
    cap.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        cs = torch.cuda.current_stream()
        s_in.wait_stream(cs)
        s_out.wait_stream(cs)
        for k in range(E2E_GRAPH):
            e2e_step(k, cs, first=k < 2)
        cs.wait_event(ev_out[(E2E_GRAPH - 1) % 2])
        cs.wait_event(ev_out[E2E_GRAPH % 2])
    stream.wait_stream(cap)
    graph.replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(reps):
        graph.replay()
    g1.record(stream)
    torch.cuda.synchronize()
    e2e_steps = reps * E2E_GRAPH
    e2e_graph_ms = max_over_ranks(g0.elapsed_time(g1), world)
    del graph
    # the line reports the faster of the two loops (both given)
    e2e_loop = "graph" if e2e_graph_ms / e2e_steps <= e2e_eager_ms / K else "eager"
    e2e_ms, e2e_steps = (e2e_graph_ms, e2e_steps) if e2e_loop == "graph" else (e2e_eager_ms, K)
    e2e_value = throughput_gbs(world, sbytes, e2e_ms / e2e_steps)
    case.q_new, case.k_new, case.v_new, case.pos, case.seq_lens = view_sets[0]
    bufs.out = outs[0]
    host_out = host_outs[0]

    # the same step with its inputs and output in the pinned host block: the
    # kernels read q, k, v, positions and lengths and write the output across
    # the CPU-GPU link themselves (GB300's coherent link; no copy launches),
    # the same bytes crossing per step
    dev_views = (case.q_new, case.k_new, case.v_new, case.pos, case.seq_lens)
    dev_out = bufs.out
    case.q_new, case.k_new, case.v_new, case.pos, case.seq_lens = [
        host_blk[o:o + x.numel() * x.element_size()].view(x.dtype).view(x.shape) for x, o in zip(dev_views, offs)]
    bufs.out = host_out
    for _ in range(3):
        step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    z0 = torch.cuda.Event(enable_timing=True)
    z1 = torch.cuda.Event(enable_timing=True)
    z0.record(stream)
    for _ in range(K):
        step()
    z1.record(stream)
    torch.cuda.synchronize()
    zc_ms = max_over_ranks(z0.elapsed_time(z1), world)
    zc_value = throughput_gbs(world, sbytes, zc_ms / K)
    case.q_new, case.k_new, case.v_new, case.pos, case.seq_lens = dev_views
    bufs.out = dev_out

    peak, peak_src = measured_peak()
    sweep = (world == 1 and args.workload == DEFAULT_WORKLOAD and args.cache == "native" and nn == 1
             and args.window == 0 and args.variant == 0 and not args.no_workloads)
    workloads = measure_workloads(m, dev, stream, max(50, K), sampler, peak) if sweep else None
    sampler.stop()
    if tc05:
        kernel_name = "attn_tc05_kernel"
    elif byte:
        heads_kernel = w.paged and w.page_size in (16, 32) and w.group <= 16 and w.h_kv % 2 == 0
        # one new token and 32 query heads per kv head on tcgen05: uint8 with
        # the keys on the MMA rows, e5m2 with the heads on the rows and the
        # codes widened by converter warps
        keys_kernel = nn == 1 and 16 < w.group <= 32 and not w.paged and w.head_dim == 128
        kernel_name = (("attn_tc05_keys_kernel" if args.cache == "u8" else "attn_tc05_widen_kernel") if keys_kernel else
                       "decode_u8_heads_kernel" if heads_kernel else "decode_u8_kernel")
    elif variant in (0, 2) and w.dtype == "bf16":
        heads_kernel = (w.paged and w.page_size == 16 and w.head_dim == 128 and w.group <= 16 and w.h_kv % 2 == 0
                        and nn == 1)
        kernel_name = "decode_mma_heads_kernel" if heads_kernel else "decode_mma_kernel"
    else:
        kernel_name = "decode_fma_kernel"
    if fused and (splits_used == 1 or merged):
        # the step is this one launch: its average duration over the timed
        # region is the step time, and it moves the whole step's bytes
        roof_bytes, roof_ms = sbytes, ms_per_step
        roof_kernel = kernel_name + " (append fused" + (", two-block clusters merging the splits)" if merged else ")")
        roof_time = "timed region: K back-to-back launches of this kernel, CUDA events at both ends"
    elif fused:
        roof_bytes, roof_ms = sbytes, step_call_ms
        roof_kernel = kernel_name + " (append fused) + combine_kernel"
        roof_time = "events around each step call (decode + combine launches)"
    else:
        roof_bytes, roof_ms = abytes, attn_ms
        roof_kernel = kernel_name + (" + combine_kernel" if splits_used > 1 and not merged else "")
        roof_time = "events around each standalone gqa_decode_attention call"
    achieved = roof_bytes / (roof_ms * 1e-3) / 1e9
    traffic = (ncu_traffic(args.workload + ("_" + args.cache if byte else "")) if kernel_name.startswith(("decode_mma", "decode_u8", "attn_tc05"))
               else None)
    clocks = sampler.summary(t_clock0, t_clock1)

    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": UNIT,
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 6),
        "us_per_step": round(ms_per_step * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": args.cache if byte else w.dtype,
        "data": ("synthetic (seeded N(0,1) bf16 q/k/v; uint8 cache codes U[0,255], scales ~6/255, zero points "
                 "U[100,155]; no dataset)" if u8 else
                 "synthetic (seeded N(0,1) bf16 q/k/v; N(0,1) cache rounded to fp8 e5m2; no dataset)" if f8 else
                 "synthetic (seeded N(0,1) bf16 q/k/v and cache; no dataset)"),
        "config": {
            "workload": (f"{w.name}: batch {w.batch}, H_q {w.h_q}, H_kv {w.h_kv}, head_dim {w.head_dim}, "
                         + (f"paged {w.page_size}-token pages, lengths U[{w.len_lo},{w.len_hi}]" if w.paged
                            else f"contiguous {'uint8' if u8 else 'fp8 e5m2' if f8 else w.dtype} cache of "
                                 f"{w.seq_len} tokens/seq")
                         + (", uint8 cache codes + float32 (scale, zero point) per row" if u8 else "")
                         + (f", {nn} new tokens per sequence verified in one pass (causal among them)"
                            if nn > 1 else "")
                         + ", RoPE base 10000"),
            "cache": args.cache if byte else w.dtype,
            "n_new": nn,
            "batch_per_gpu": w.batch,
            "tokens_per_step_per_gpu": int(lens_cpu.sum()),
            "num_splits": splits_used,
            "window": args.window,
            "variant": {0: "auto", 1: "cuda_core", 2: "tensor_core"}[variant],
            "bytes_per_step_per_gpu": sbytes,
            "l2": "inputs larger than L2 (no flush): %.0f MB streamed per step vs 129 MB L2" % (sbytes / 1e6),
            "parallelism": f"dp{world}" if world > 1 else "single",
        },
        "kernels_ms": {"mqa_decode_step": round(step_call_ms, 6),
                       "standalone_kv_append_rope": round(append_ms, 6),
                       "standalone_gqa_decode_attention": round(attn_ms, 6),
                       "how": "CUDA events around each call on the launching stream, second pass of the same steps"},
        "roofline": {
            "bound": "hbm",
            "kernel": roof_kernel,
            "achieved": round(achieved, 2),
            "peak": peak,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": traffic,
            "algorithmic_bytes_per_launch": roof_bytes,
            "duration_ms": round(roof_ms, 6),
            "duration_from": roof_time,
            "peak_source": peak_src,
            "frac_of_8000": round(achieved / 8000.0, 4),
        },
        "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms / e2e_steps, 6), "steps": e2e_steps, "loop": e2e_loop,
                "graph_ms_per_step": round(e2e_graph_ms / (reps * E2E_GRAPH), 6),
                "eager_ms_per_step": round(e2e_eager_ms / K, 6),
                "how": "each step: one cudaMemcpyAsync of its packed pinned inputs (a copy stream, overlapping the "
                       "previous step; double-buffered device block), the step through the C ABI, one "
                       "cudaMemcpyAsync of its output (a second copy stream, overlapping the next step); the loop "
                       "issued from Python every step (eager) and as 32 such steps captured once into a CUDA "
                       "graph and replayed (graph); value = the faster of the two, named in loop"},
        "e2e_host_io": {"value": round(zc_value, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
                        "d2h_bytes_per_step": d2h, "ms_per_step": round(zc_ms / K, 6),
                        "how": "each step: the kernels read the inputs from and write the output to pinned host "
                               "memory across the CPU-GPU link (no copy launches)"},
        "gpu_launches": K * launches_per_step,
        "clocks": clocks,
    }
    if workloads is not None:
        line["workloads"] = workloads

    if do_cpu:
        single, multi, outs = oracle_baseline(w, units, out_es, args.cache, nn, args.window, args.cpu_seconds)
        out_host = bufs.out.float().cpu().numpy()
        G = w.group
        if nn > 1:
            errs = [float(np.max(np.abs(out_host[u["b"], :, u["j"] * G:(u["j"] + 1) * G] - o)))
                    for u, o in zip(units, outs)]
        else:
            errs = [float(np.max(np.abs(out_host[u["b"], u["j"] * G:(u["j"] + 1) * G] - o)))
                    for u, o in zip(units, outs)]
        per_unit_ms = 1e3 * statistics.fmean(unit_bytes(w, u["L"], out_es, args.cache, nn) for u in units) / (
            multi["value"] * 1e9)
        line["cpu_baseline"] = {
            "value": round(multi["value"], 6), "unit": UNIT, "cores": multi["cores"], "kind": "oracle",
            "sample": f"{len(units)} distinct (sequence, kv head) units of the step (of {w.batch * w.h_kv}), "
                      f"fp64 numpy, one single-threaded process per host core cycling over its share of them; "
                      f"median of {len(multi['runs_gbs'])} runs of {args.cpu_seconds:.1f} s",
            "runs_gbs": [round(x, 6) for x in multi["runs_gbs"]],
            "single_thread": {"value": round(single["value"], 6), "unit": UNIT, "cores": 1,
                              "runs_gbs": [round(x, 6) for x in single["runs_gbs"]],
                              "sample": f"the same units in one thread, median of {len(single['runs_gbs'])} runs "
                                        f"of {args.cpu_seconds:.1f} s"},
            "ms_per_step_extrapolated": round(sbytes / (multi["value"] * 1e9) * 1e3, 1),
            "ms_per_unit_all_cores": round(per_unit_ms, 3),
        }
        line["parity_sample"] = {"units": len(units), "max_abs_err": max(errs), "tolerance": 2e-2}
        if workloads is not None:
            line["workloads"]["tiny"] = tiny_parity(m, dev)

    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# ------------------------------------------------------------ prefill leg
PREFILL_METRIC = "prefill causal attention TFLOP/s (fraction of GB300 bf16 peak) at 1 GPU"


def prefill_flops(w, n):
    """Algorithmic FLOPs of causal attention over n new tokens per sequence
    (no prefix): query i scores and mixes i + 1 keys, 4 d FLOPs per (head, key)."""
    return 4 * w.head_dim * w.h_q * w.batch * n * (n + 1) // 2


def bench_prefill(args):
    """The prompt's tokens appended and attended causally in one pass
    (mqa_prefill_step): time per step and the attention kernel's TFLOP/s."""
    import mqa_decode_attention_gb300 as m

    world, rank, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    n = args.prefill
    w = workload(args.workload).with_(batch=args.batch or 8)
    full = torch.full((w.batch,), n, dtype=torch.int32)
    if w.paged:  # the prompt's rows go to the pages the (permuted) block table names
        pc = make_paged_case(w, dev, seq_lens=full)
        rows_shape, lens, table = (pc.num_pages, w.h_kv, pc.page_size), pc.seq_lens, pc.block_table
        kb, vb = pc.k_pool, pc.v_pool
    else:
        case = make_contiguous_case(w, dev, seq_lens=full, capacity=n)
        rows_shape, lens, table = (w.batch, w.h_kv, n), case.seq_lens, None
        kb, vb = case.k_cache, case.v_cache
    extra = {}
    if args.cache == "u8":  # codes with per-row (scale, zero point)
        u = make_u8_cache(rows_shape, w.head_dim, w.seed + 5, dev)
        kb, vb = u.k_codes, u.v_codes
        extra = dict(k_scale_zero=u.k_sz, v_scale_zero=u.v_sz)
    elif args.cache == "fp8":
        kb, vb = make_e5m2_cache(rows_shape, w.head_dim, w.seed + 5, dev)
    lay = (m.layout_paged(kb, vb, table, w.h_q, **extra) if w.paged else
           m.layout_contiguous(kb, vb, w.h_q, **extra))
    q = normal((w.batch, n, w.h_q, w.head_dim), w.seed, S_QM, w.dtype, dev)
    k = normal((w.batch, n, w.h_kv, w.head_dim), w.seed, S_KM, w.dtype, dev)
    v = normal((w.batch, n, w.h_kv, w.head_dim), w.seed, S_VM, w.dtype, dev)
    bufs = m.DecodeBuffers.allocate(lay, n, num_splits=1, device=dev, n_new=n)
    pos = (lens - n).to(torch.int32)
    scale = 1.0 / math.sqrt(w.head_dim)
    stream = torch.cuda.current_stream()

    def step():
        m.prefill_step(lay, n, q, k, v, pos, lens, n, bufs, w.rope_base, scale, stream)

    sampler = ClockSampler(gpu_index_for(local))
    t_warm = time.monotonic()
    n_warm = 0
    while n_warm < args.warmup or time.monotonic() - t_warm < args.warm_seconds:
        step()
        n_warm += 1
    torch.cuda.synchronize()
    t_clock0 = time.monotonic() - 0.5
    K = args.steps
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(K):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms_step = e0.elapsed_time(e1) / K
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * K)]
    for i in range(K):
        ev[2 * i].record(stream)
        m.gqa_prefill_attention(lay, n, bufs.q_rot, lens, n, scale, bufs.out, bufs.lse, bufs.err, stream)
        ev[2 * i + 1].record(stream)
    torch.cuda.synchronize()
    t_clock1 = time.monotonic()
    sampler.stop()
    attn_ms = statistics.fmean(ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(K))
    if int(bufs.err.item()) != 0:
        raise RuntimeError(f"device error word {int(bufs.err.item()):#x}")
    flops = prefill_flops(w, n)
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except (OSError, ValueError):
        pass
    peak = float(peaks.get("bf16_tflops", 1900.0))
    achieved = flops / (attn_ms * 1e-3) / 1e12
    line = {
        "metric": PREFILL_METRIC,
        "value": round(flops / (ms_step * 1e-3) / 1e12, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 6),
        "higher_is_better": True,
        "dtype": {"native": "bf16", "u8": "u8", "fp8": "fp8_e5m2"}[args.cache],
        "data": "synthetic (seeded N(0,1) bf16 q/k/v; " + {"native": "bf16", "u8": "uint8", "fp8": "fp8 e5m2"}[args.cache]
                + " cache, empty before the prompt)",
        "config": {"workload": f"prefill: batch {w.batch}, {n}-token prompts, H_q {w.h_q}, H_kv {w.h_kv}, "
                               f"head_dim {w.head_dim}, causal, RoPE base 10000, "
                               + (f"paged pool (page_size {w.page_size}, pages dealt by a seeded permutation)"
                                  if w.paged else "contiguous cache")
                               + {"native": ", bf16", "u8": ", uint8 codes + (scale, zero point)", "fp8": ", fp8 e5m2"}[args.cache],
                   "flops_per_step": flops},
        "kernels_ms": {"mqa_prefill_step": round(ms_step, 6), "standalone_gqa_prefill_attention": round(attn_ms, 6)},
        "roofline": {"bound": "tensor",
                     "kernel": ("attn_tc05_prefill_kernel" if args.cache == "native" else
                                "decode_u8_kernel (multi-token form)" if args.cache == "u8" or w.paged else
                                "attn_tc05_prefill_kernel (fp8 form)"),
                     "achieved": round(achieved, 1),
                     "peak": peak, "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": None,
                     "peak_source": "MEASURED_PEAKS.json bf16_tflops (cuBLAS burst)" if peaks else "fallback"},
        "gpu_launches": 2 * K,
        "clocks": sampler.summary(t_clock0, t_clock1),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


# ---------------------------------------------------------- reference arm
def bench_reference(args):
    from oracle import cores  # test infrastructure: the reference (oracle) arm only

    world, rank, _ = dist_env()
    if rank != 0:
        return
    w = workload(args.workload)
    case = build_case(w, "cpu", args.cache, args.n_new)
    lens = case.seq_lens
    n_units = w.batch * w.h_kv
    order = [(u // w.h_kv, u % w.h_kv) for u in range(n_units)]
    out_es = 4 if w.dtype == "f32" else 2
    meta = oracle_meta(w, args.window)
    picked = order[:min(n_units, args.warmup + args.steps)]
    inputs = [cores.widen(u, meta) for u in numpy_units(w, unit_inputs(w, case, picked), out_es, args.cache,
                                                        args.n_new, args.window)]

    def run(i):
        u = inputs[i % len(inputs)]
        cores.run_unit(u, meta)
        return int(u["bytes"])

    for i in range(args.warmup):
        run(i)
    t0 = time.perf_counter()
    done = 0
    for i in range(args.steps):
        done += run(args.warmup + i)
    secs = time.perf_counter() - t0
    value = done / secs / 1e9
    line = {
        "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(secs / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1) bf16 inputs)",
        "impl": "reference",
        "config": {"workload": w.name, "cache": args.cache if args.cache in ("u8", "fp8") else w.dtype,
                   "window": args.window,
                   "n_new": args.n_new,
                   "batch_per_gpu": w.batch, "tokens_per_step_per_gpu": int(lens.sum()),
                   "step": "one (sequence, kv head) unit of the workload per step, cycling over the units"},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{args.steps} units of {n_units}, fp64 numpy, single thread"},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--splits", type=int, default=None, help="override the workload's split count (0 = auto)")
    ap.add_argument("--variant", type=int, default=0, help="0 auto, 1 CUDA cores, 2 tensor cores")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the L2-controlled pass over every workload (the default bench line carries it)")
    ap.add_argument("--warm-seconds", type=float, default=1.0,
                    help="minimum warm-up time, so the clock sampler sees the load (0 for profiler runs)")
    ap.add_argument("--batch", type=int, default=0, help="override the workload's batch (smaller profiling cases)")
    ap.add_argument("--window", type=int, default=0, help="sliding window: attend to the last W tokens (0 = all)")
    ap.add_argument("--prefill", type=int, default=0,
                    help="time prefill of this many prompt tokens per sequence instead of a decode step")
    ap.add_argument("--n-new", type=int, default=1,
                    help="new tokens per sequence (the verification pass of speculative decoding)")
    ap.add_argument("--cache", choices=["native", "u8", "fp8"], default="native",
                    help="cache type: the workload's own (bf16 / fp32) or uint8 codes with per-row scale / zero point")
    ap.add_argument("--cpu-seconds", type=float, default=3.0, help="seconds per oracle timing run (3 runs each)")
    ap.add_argument("--cpu-units", type=int, default=0, help="distinct units in the CPU sample (0 = all)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        bench_reference(args)
    elif args.prefill:
        bench_prefill(args)
    else:
        bench_ours(args)


if __name__ == "__main__":
    main()
