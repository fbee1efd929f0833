"""The log-sum-exp each decode kernel forms, modelled in fp64 from the
oracle's rotated query, so that the kernels' fp32 lse outputs can be held to
fp32 accuracy instead of the bf16 output tolerance.

Every kernel multiplies q_rot by c = fp32(scale * log2 e) in fp32 and rounds
the product to its MMA operand type before the scores are formed: bf16 on the
bf16-cache tensor-core kernels (warp MMA and tcgen05), fp16 on the warp-MMA
e5m2-cache kernels, none on the CUDA-core (fp32) path; the tcgen05 e5m2-cache
kernel takes x = q c 2^6 as two e4m3 values hi = e4m3(x), lo = e4m3(x - hi)
(fmt "e4m3x2"). That one rounding moves a score by
up to 2^-8 of the sum of its terms' magnitudes for bf16 (about 1e-3 on N(0,1)
data at d = 128), far more than everything after it: fp32 accumulation, the
ex2 approximation, the split combine. The model applies the same rounding to
the oracle's fp64 q_rot and takes the log-sum-exp of the resulting scores in
fp64, so what remains between it and the GPU is fp32 arithmetic: LSE_TOL.

The GPU's own q_rot comes from an fp32 rotation (relative error below 1e-6 of
the fp64 one), so an element of q * c lying within that distance of a rounding
boundary may round the other way on the GPU. Such elements widen their row's
tolerance by what that change of the operand can move the log-sum-exp (it is
1-Lipschitz in the largest score change): ln 2 * |change| * max_t |k_t,i|.
"""

import math

import numpy as np
import torch

import oracle

LSE_TOL = 1e-4
_LOG2E = np.float32(1.4426950408889634)
_AMBIGUOUS = 2e-6  # relative distance to a rounding boundary that the fp32 rotation may cross


def _e4m3(x: np.ndarray) -> np.ndarray:
    """Round to e4m3 (nearest, ties to even), saturating at 448."""
    t = torch.from_numpy(np.clip(np.ascontiguousarray(x, np.float32), -448.0, 448.0))
    return t.to(torch.float8_e4m3fn).to(torch.float32).numpy()


def _round(x32: np.ndarray, fmt: str) -> np.ndarray:
    if fmt == "e4m3x2":
        x = x32.astype(np.float32) * np.float32(64.0)
        hi = _e4m3(x)
        lo = _e4m3((x - hi).astype(np.float32))
        return (hi.astype(np.float64) + lo.astype(np.float64)) / 64.0
    if fmt == "bf16":
        return torch.from_numpy(np.ascontiguousarray(x32)).to(torch.bfloat16).to(torch.float64).numpy()
    if fmt == "f16":
        return x32.astype(np.float16).astype(np.float64)
    if fmt == "f32":
        return x32.astype(np.float64)
    raise ValueError(fmt)


def model_lse(q_rot, keys, lens, scale: float, fmt: str, window: int = 0, key_scales=None):
    """q_rot [B, H_q, d] or [B, n, H_q, d] (the oracle's, fp64); keys [B, H_kv,
    T, d] (the logical cache after the append, the values the kernel reads);
    lens [B] after the append, new token i of n at position L - n + i.
    key_scales [B, H_kv, T] (uint8 caches): the per-row scales s_t of the keys,
    for the zero-point cancellation bound below.
    Returns (lse, tol), each shaped like q_rot without its last axis."""
    q = np.asarray(q_rot, np.float64)
    single = q.ndim == 3
    if single:
        q = q[:, None]
    keys = np.asarray(keys, np.float64)
    lens = np.asarray(lens).astype(np.int64)
    B, n, h_q, d = q.shape
    h_kv = keys.shape[1]
    G = h_q // h_kv
    c = np.float32(scale) * _LOG2E
    qs = (q.astype(np.float32) * c).astype(np.float32)
    qr = _round(qs, fmt)
    if fmt == "f32":
        spread = np.zeros_like(qr)
    else:
        # how far the operand moves when q c moves by the fp32 rotation's error
        lo = _round((qs.astype(np.float64) * (1 - _AMBIGUOUS)).astype(np.float32), fmt)
        hi = _round((qs.astype(np.float64) * (1 + _AMBIGUOUS)).astype(np.float32), fmt)
        spread = np.maximum(np.abs(lo - qr), np.abs(hi - qr))
    lse = np.empty((B, n, h_q))
    tol = np.empty((B, n, h_q))
    for b in range(B):
        L = int(lens[b])
        for i in range(n):
            end = L - n + i + 1
            t0 = oracle.window_start(end, window)
            for j in range(h_kv):
                K = keys[b, j, t0:end]                     # [T, d]
                rows = slice(j * G, (j + 1) * G)
                s = (K @ qr[b, i, rows].T) * math.log(2.0)  # [T, G]
                m = s.max(axis=0)
                lse[b, i, rows] = m + np.log(np.exp(s - m).sum(axis=0))
                tol[b, i, rows] = LSE_TOL + math.log(2.0) * (spread[b, i, rows] @ np.abs(K).max(axis=0))
                if key_scales is not None:
                    tol[b, i, rows] += _u8_cancellation(qr[b, i, rows], key_scales[b, j, t0:end], d)
    if single:
        lse, tol = lse[:, 0], tol[:, 0]
    return lse, tol


def _u8_cancellation(qr, s_k, d: int) -> np.ndarray:
    """Bound (natural-log units) on the fp32 error of a uint8-cache score formed
    as s_t (sum_d q_d (1024 + c_td) - (1024 + z_t) sum_d q_d), the warp-MMA
    kernel's form: the MMA's fp32 partial sums (d / 16 k-steps) and the
    subtraction, each at most 1279 sum_d |q_d| in magnitude, round with
    relative error <= 2^-23 (twice round-to-nearest's, for the tensor core's
    accumulation); the fp32 row sum of q loses <= d 2^-24 sum_d |q_d| before it
    is multiplied by 1024 + z_t <= 1279. Every term scales with s_t."""
    mag = 1279.0 * np.abs(qr).sum(axis=-1)
    return math.log(2.0) * float(np.max(s_k)) * mag * (d / 16 + 2 + d / 2) * 2.0 ** -23


def paged_keys(pool, table, lens, page_size: int) -> np.ndarray:
    """The logical keys [B, H_kv, max L, d] of a paged pool (zeros past each length)."""
    pool = np.asarray(pool, np.float64)
    table = np.asarray(table).astype(np.int64)
    lens = np.asarray(lens).astype(np.int64)
    out = np.zeros((len(lens), pool.shape[1], int(lens.max()), pool.shape[-1]))
    for b, L in enumerate(lens):
        out[b, :, :L] = oracle.gather_paged(pool, table[b], int(L), page_size)
    return out


def assert_lse(got, q_rot, keys, lens, scale: float, fmt: str, window: int = 0, what=None, key_scales=None):
    """The GPU's lse within LSE_TOL (plus the per-row widening above) of the model."""
    ref, tol = model_lse(q_rot, keys, lens, scale, fmt, window, key_scales)
    got = np.asarray(got, np.float64).reshape(ref.shape)
    err = np.abs(got - ref)
    worst = np.unravel_index(np.argmax(err - tol), err.shape)
    assert np.all(err <= tol), (what, worst, float(err[worst]), float(tol[worst]))
