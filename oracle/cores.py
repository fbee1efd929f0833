"""The oracle's decode step on every host core -- TEST INFRASTRUCTURE.

Only bench.py's CPU-baseline leg uses this module. It runs the oracle's own
per-(sequence, kv head) decode step -- ``decode_unit`` for a bf16 / fp32
cache, ``decode_step_u8`` and ``decode_step_e5m2`` for the one-byte caches,
``decode_step_multi`` for several new tokens -- over a sample of units, one
single-threaded process per core (numpy's BLAS pinned to one thread each),
the units spread over the processes. The arithmetic is the oracle's as it
stands; nothing here blocks, fuses or reorders it.

    python -m oracle.cores UNITS.npz --seconds S --runs R --procs P

reads the units written by ``save_units`` and prints one JSON line: for each
run, the bytes and units done by all processes together and the wall time
from a common start to the last process's end.
"""

from __future__ import annotations

import argparse
import json
import os
import time

for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import numpy as np  # noqa: E402

from . import decode  # noqa: E402

_FLOAT_FIELDS = ("q", "k", "v", "K", "V")
_RAW_FIELDS = ("Kc", "Ks", "Vc", "Vs", "K8", "V8")


def _bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 values stored as their 16-bit patterns, widened exactly."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def save_units(path: str, units: list[dict], meta: dict) -> None:
    """Write units (dicts of numpy arrays; float fields either float32 or the
    uint16 bit patterns of bf16 values, flagged by meta["bf16_bits"]) and the
    step's parameters to an .npz file."""
    arrays = {"meta": np.array(json.dumps(meta))}
    for i, u in enumerate(units):
        for key, val in u.items():
            arrays[f"u{i}_{key}"] = np.asarray(val)
    arrays["count"] = np.array(len(units))
    np.savez(path, **arrays)


def widen(raw: dict, meta: dict) -> dict:
    """A unit as save_units takes it, float fields widened to float64."""
    u = {}
    for key, val in raw.items():
        val = np.asarray(val)
        if key in _FLOAT_FIELDS:
            val = _bits_to_f64(val) if meta["bf16_bits"] else val.astype(np.float64)
        elif key not in _RAW_FIELDS:
            val = val.item() if val.ndim == 0 else val
        u[key] = val
    return u


def load_units(path: str, indices=None):
    """The units of an .npz file written by save_units, float fields widened to
    float64. Returns (units, meta)."""
    z = np.load(path)
    meta = json.loads(str(z["meta"]))
    count = int(z["count"])
    units = []
    for i in (range(count) if indices is None else indices):
        prefix = f"u{i}_"
        units.append(widen({name[len(prefix):]: z[name] for name in z.files if name.startswith(prefix)}, meta))
    return units, meta


def run_unit(u: dict, meta: dict) -> np.ndarray:
    """The oracle's decode step for one (sequence, kv head) unit: its output rows."""
    scale, base, window, dtype = meta["scale"], meta["rope_base"], meta["window"], meta["dtype"]
    L = int(u["L"])
    if "K8" in u:
        r = decode.decode_step_e5m2(u["K8"][None, None], u["V8"][None, None], u["q"][None], u["k"][None, None],
                                    u["v"][None, None], [L], base, scale, window=window)
        return r["out"][0]
    if "Kc" in u:
        r = decode.decode_step_u8(u["Kc"][None, None], u["Ks"][None, None], u["Vc"][None, None], u["Vs"][None, None],
                                  u["q"][None], u["k"][None, None], u["v"][None, None], [L], base, scale,
                                  window=window)
        return r["out"][0]
    if int(u["n"]) > 1:
        r = decode.decode_step_multi(u["K"][None, None], u["V"][None, None], u["q"][None], u["k"][None, :, None],
                                     u["v"][None, :, None], [L], base, scale, dtype, window=window)
        return r["out"][0]
    o, _, _ = decode.decode_unit(u["q"], u["k"], u["v"], u["K"], u["V"], L, base, scale, dtype, window=window)
    return o


def run_for(units: list[dict], meta: dict, seconds: float, start: float | None = None):
    """Cycle through the units until `seconds` have passed (at least one unit).
    Returns (bytes done, units done, elapsed seconds)."""
    if start is not None:
        while time.time() < start:
            time.sleep(0.001)
    t0 = time.perf_counter()
    done = nbytes = 0
    i = 0
    while True:
        u = units[i % len(units)]
        run_unit(u, meta)
        nbytes += int(u["bytes"])
        done += 1
        i += 1
        if time.perf_counter() - t0 >= seconds:
            break
    return nbytes, done, time.perf_counter() - t0


_CACHE: dict = {}


def _worker(path: str, indices: list[int], start: float, seconds: float):
    key = (path, tuple(indices))
    if key not in _CACHE:
        _CACHE.clear()
        _CACHE[key] = load_units(path, indices)
    units, meta = _CACHE[key]
    nbytes, done, _ = run_for(units, meta, seconds, start)
    return nbytes, done, time.time()


def main() -> None:
    import multiprocessing as mp

    ap = argparse.ArgumentParser()
    ap.add_argument("path")
    ap.add_argument("--seconds", type=float, default=3.0)
    ap.add_argument("--runs", type=int, default=3)
    ap.add_argument("--procs", type=int, default=0)
    args = ap.parse_args()
    procs = args.procs or len(os.sched_getaffinity(0))
    count = int(np.load(args.path)["count"])
    shares = [[i for i in range(count) if i % procs == p] or [p % count] for p in range(procs)]
    runs = []
    with mp.get_context("spawn").Pool(procs) as pool:
        pool.starmap(_worker, [(args.path, s, 0.0, 0.0) for s in shares])  # load the units, warm up
        for _ in range(args.runs):
            start = time.time() + 0.5
            res = pool.starmap(_worker, [(args.path, s, start, args.seconds) for s in shares])
            wall = max(r[2] for r in res) - start
            runs.append({"bytes": sum(r[0] for r in res), "units": sum(r[1] for r in res), "wall_s": wall})
    print(json.dumps({"procs": procs, "runs": runs}), flush=True)


if __name__ == "__main__":
    main()
