"""Seeded synthetic workloads for the verification step.

Shared by the tests, the bench and the smoke check.  This module holds none of
the method's arithmetic: it draws random numbers (``synth.c``, SplitMix64
counters) and lays them out the way ``sd_plan`` / ``sd_verify`` consume them.
Random numbers the method itself uses (the acceptance uniforms) are drawn here
and passed in as inputs, so the oracle and the CUDA path see identical bytes.

Workloads (shapes and distributions of the pages' serving setups; synthetic
stand-ins for the pages' MT-Bench and in-house traffic, which are not used):

  tiny          BS=4,    K=3, V=1024,   fp32  target N(0,2^2), draft +N(0,0.5^2)
  dense_fixed_k BS=64,   K=3, V=256000, bf16  target N(0,3^2), draft +N(0,1), all slots
  adaptive_hc   BS=256,  K=7, V=129280, bf16  draft noise sd 0.5 -> 2.0 with position
  varlen_mixed  BS=128,  K_i in 1..7,  V=129280, fp32, 20 steps, budget from step t-1
  stress        BS=1024, K=7, V=129280, bf16  draft noise sd 1.5
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass, field, replace
from pathlib import Path
from typing import Callable, Optional

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "synth.c"
_LIB = _HERE / "libsdsynth.so"

F32, BF16 = 0, 1
MODE_ADAPTIVE, MODE_ALL_SLOTS, MODE_UNIFORM_K = 0, 1, 2
ST_CONF, ST_UNIFORM, ST_LENS = 10, 11, 12


def build(force: bool = False) -> Path:
    if force or not _LIB.exists() or _LIB.stat().st_mtime < _SRC.stat().st_mtime:
        tmp = _LIB.with_suffix(f".so.tmp{os.getpid()}")
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                        "-Wall", "-o", str(tmp), str(_SRC), "-lm", "-lpthread"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(str(_LIB))
        P, u64, i64, i32 = ctypes.c_void_p, ctypes.c_uint64, ctypes.c_int64, ctypes.c_int32
        lib.synth_logit_rows.argtypes = [u64, u64, i64, P, P, i32, i32, ctypes.c_double, P, P,
                                         ctypes.c_int]
        lib.synth_draft_ids.argtypes = [u64, u64, i64, P, P, P, i32, i32, P, P, ctypes.c_int]
        lib.synth_uniforms.argtypes = [u64, u64, u64, i64, P, P, P]
        lib.synth_normals.argtypes = [u64, u64, u64, i64, P, P, P]
        for f in (lib.synth_logit_rows, lib.synth_draft_ids, lib.synth_uniforms, lib.synth_normals):
            f.restype = ctypes.c_int
        _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _threads():
    return max(1, min(64, os.cpu_count() or 1))


def logit_rows(seed, step, req, pos, V, dtype, sigma_t, sigma_d=None):
    """Rows [len(req), V]: fp32 array, or uint16 bf16 bit patterns."""
    req = np.ascontiguousarray(req, np.int32)
    pos = np.ascontiguousarray(pos, np.int32)
    out = np.empty((len(req), V), np.float32 if dtype == F32 else np.uint16)
    sd = None if sigma_d is None else np.ascontiguousarray(sigma_d, np.float64)
    rc = _load().synth_logit_rows(seed, step, len(req), _p(req), _p(pos), V, dtype,
                                  float(sigma_t), _p(sd), _p(out), _threads())
    if rc != 0:
        raise ValueError("synth_logit_rows failed")
    return out


def draft_ids(seed, step, req, pos, rows, V, dtype, tau):
    req = np.ascontiguousarray(req, np.int32)
    pos = np.ascontiguousarray(pos, np.int32)
    tau = np.ascontiguousarray(tau, np.float32)
    rows = np.ascontiguousarray(rows)
    ids = np.zeros(len(req), np.int32)
    rc = _load().synth_draft_ids(seed, step, len(req), _p(req), _p(pos), _p(rows), V, dtype,
                                 _p(tau), _p(ids), _threads())
    if rc != 0:
        raise ValueError("synth_draft_ids failed")
    return ids


def uniforms(seed, stream, step, i, j):
    i = np.ascontiguousarray(i, np.int32)
    j = np.ascontiguousarray(j, np.int32)
    out = np.zeros(len(i), np.float32)
    if _load().synth_uniforms(seed, stream, step, len(i), _p(i), _p(j), _p(out)) != 0:
        raise ValueError("synth_uniforms failed")
    return out


def normals(seed, stream, step, i, j):
    i = np.ascontiguousarray(i, np.int32)
    j = np.ascontiguousarray(j, np.int32)
    out = np.zeros(len(i), np.float64)
    if _load().synth_normals(seed, stream, step, len(i), _p(i), _p(j), _p(out)) != 0:
        raise ValueError("synth_normals failed")
    return out


# ----------------------------------------------------------------------------
# Cost tables (step cost by token count n = T + B)


def ceil_to(n, m):
    return m * ((n + m - 1) // m)


def cost_linear_stairs(a, b, stair, nmax):
    """cost(n) = a + b * ceil_stair(n) for n = 0..nmax."""
    n = np.arange(nmax + 1)
    return (a + b * ceil_to(n, stair)).astype(np.float32)


# CUDA-graph capture sizes of the varlen workload: the listed start
# {1,2,4,8,16,24,32,48,64,...,1024}, continued with the x1.5 / x2 pattern.
GRAPH_SIZES = (1, 2, 4, 8, 16, 24, 32, 48, 64, 96, 128, 192, 256, 384, 512, 768, 1024)


def cost_graph_sizes(a, b, sizes=GRAPH_SIZES):
    """cost(n) = a + b * g(n), g(n) = smallest captured size >= n, n = 0..max."""
    nmax = sizes[-1]
    s = np.asarray(sizes)
    n = np.arange(nmax + 1)
    g = s[np.searchsorted(s, n, side="left")]
    return (a + b * g).astype(np.float32)


# ----------------------------------------------------------------------------
# Workload definitions


@dataclass(frozen=True)
class Workload:
    name: str
    bs: int
    k_max: int
    V: int
    dtype: int
    sigma_t: float
    sigma_d: Callable[[np.ndarray, np.ndarray], np.ndarray]  # (pos j, K_i) -> sd
    temps: Callable[[int], np.ndarray]
    mode: int = MODE_ADAPTIVE
    conf_mean: Optional[Callable[[np.ndarray], np.ndarray]] = None
    conf_sd: float = 1.0
    T: int = 0
    cost: Optional[np.ndarray] = None
    varlen: bool = False  # K_i ~ U{1..k_max} per step
    steps: int = 1
    budget_from_previous: bool = False

    @property
    def elem(self):
        return 4 if self.dtype == F32 else 2

    def with_(self, **kw):
        return replace(self, **kw)


def _temps_cycle(values):
    v = np.asarray(values, np.float32)
    return lambda bs: v[np.arange(bs) % len(v)]


def _sigma_rising(j, K):
    K = np.maximum(np.asarray(K), 2)
    return 0.5 + 1.5 * np.asarray(j) / (K - 1)


WORKLOADS = {
    "tiny": Workload(
        name="tiny", bs=4, k_max=3, V=1024, dtype=F32, sigma_t=2.0,
        sigma_d=lambda j, K: np.full(np.shape(j), 0.5),
        temps=lambda bs: np.where(np.arange(bs) < bs // 2, 0.0, 1.0).astype(np.float32),
        conf_mean=lambda j: 1.5 - 0.8 * j, conf_sd=1.0, T=4,
        cost=cost_linear_stairs(1.0, 0.01, 8, 64)),
    "dense_fixed_k": Workload(
        name="dense_fixed_k", bs=64, k_max=3, V=256000, dtype=BF16, sigma_t=3.0,
        sigma_d=lambda j, K: np.full(np.shape(j), 1.0),
        temps=_temps_cycle([1.0]), mode=MODE_ALL_SLOTS),
    "adaptive_hc": Workload(
        name="adaptive_hc", bs=256, k_max=7, V=129280, dtype=BF16, sigma_t=3.0,
        sigma_d=_sigma_rising, temps=_temps_cycle([0.0, 0.7, 1.0]),
        conf_mean=lambda j: 2.0 - 0.6 * j, conf_sd=0.7, T=256,
        cost=cost_linear_stairs(1.0, 0.004, 16, 2048)),
    "varlen_mixed": Workload(
        name="varlen_mixed", bs=128, k_max=7, V=129280, dtype=F32, sigma_t=3.0,
        sigma_d=_sigma_rising, temps=_temps_cycle([0.0, 0.7, 1.0]),
        conf_mean=lambda j: 2.0 - 0.6 * j, conf_sd=0.7, T=128,
        cost=cost_graph_sizes(1.0, 0.006), varlen=True, steps=20, budget_from_previous=True),
    "stress": Workload(
        name="stress", bs=1024, k_max=7, V=129280, dtype=BF16, sigma_t=3.0,
        sigma_d=lambda j, K: np.full(np.shape(j), 1.5), temps=_temps_cycle([1.0]),
        conf_mean=lambda j: 2.0 - 0.6 * j, conf_sd=1.0, T=1024,
        cost=cost_linear_stairs(1.0, 0.003, 32, 8192)),
}
# adaptive_hc's requests planned with one draft length for the whole batch
WORKLOADS["uniform_hc"] = WORKLOADS["adaptive_hc"].with_(name="uniform_hc", mode=MODE_UNIFORM_K)

WORKLOAD_ORDER = ("tiny", "dense_fixed_k", "adaptive_hc", "varlen_mixed", "stress")


def draft_lens(w: Workload, seed: int, step: int) -> np.ndarray:
    if not w.varlen:
        return np.full(w.bs, w.k_max, np.int32)
    i = np.arange(w.bs, dtype=np.int32)
    u = uniforms(seed, ST_LENS, step, i, np.zeros_like(i))
    return (1 + np.floor(u.astype(np.float64) * w.k_max)).astype(np.int32)


def plan_inputs(w: Workload, seed: int, step: int = 0) -> dict:
    """Inputs of sd_plan for one step: packed conf logits, draft lens, cost
    table, T, mode, plus the previous step's confidences when the workload
    sizes its budget from them (step > 0)."""
    dl = draft_lens(w, seed, step)
    out = {"draft_lens": dl, "bs": w.bs, "k_max": w.k_max, "T": w.T, "mode": w.mode,
           "cost": w.cost, "conf": None, "budget_conf": None, "budget_draft_lens": None}
    if w.mode != MODE_ALL_SLOTS:
        out["conf"] = conf_logits(w, seed, step, dl)
        if w.budget_from_previous and step > 0:
            pdl = draft_lens(w, seed, step - 1)
            out["budget_conf"] = conf_logits(w, seed, step - 1, pdl)
            out["budget_draft_lens"] = pdl
    return out


def conf_logits(w: Workload, seed: int, step: int, dl: np.ndarray) -> np.ndarray:
    i = np.repeat(np.arange(w.bs, dtype=np.int32), dl)
    j = np.concatenate([np.arange(k, dtype=np.int32) for k in dl]) if len(i) else np.zeros(0, np.int32)
    z = normals(seed, ST_CONF, step, i, j)
    return (w.conf_mean(j.astype(np.float64)) + w.conf_sd * z).astype(np.float32)


def verify_inputs(w: Workload, seed: int, step: int, cu_seqlens, draft_lens_arr,
                  requests=None) -> dict:
    """Compacted inputs of sd_verify for the plan given by cu_seqlens.

    Target row of (i, j), j = 0..n_i, sits at cu_seqlens[i] + j; draft row and
    draft id of (i, j), j < n_i, at cu_seqlens[i] - i + j.  With ``requests``
    only those requests' rows are generated (others stay zero), which lets a
    test build the rows it samples at full size cheaply."""
    cu = np.asarray(cu_seqlens, np.int64)
    bs = len(cu) - 1
    n = (cu[1:] - cu[:-1] - 1).astype(np.int64)
    temps = w.temps(bs).astype(np.float32)
    sel = np.arange(bs) if requests is None else np.asarray(sorted(set(int(r) for r in requests)))
    rows_t, rows_d = int(cu[-1]), int(cu[-1]) - bs
    tdt = np.float32 if w.dtype == F32 else np.uint16
    target = np.zeros((rows_t, w.V), tdt)
    draft = np.zeros((max(rows_d, 0), w.V), tdt)
    ids = np.zeros(max(rows_d, 0), np.int32)
    req_t = np.concatenate([np.full(n[i] + 1, i) for i in sel]).astype(np.int32)
    pos_t = np.concatenate([np.arange(n[i] + 1) for i in sel]).astype(np.int32)
    at_t = np.concatenate([cu[i] + np.arange(n[i] + 1) for i in sel])
    target[at_t] = logit_rows(seed, step, req_t, pos_t, w.V, w.dtype, w.sigma_t)
    nd = [i for i in sel if n[i] > 0]
    if nd:
        K = np.asarray(draft_lens_arr)
        req_d = np.concatenate([np.full(n[i], i) for i in nd]).astype(np.int32)
        pos_d = np.concatenate([np.arange(n[i]) for i in nd]).astype(np.int32)
        at_d = np.concatenate([cu[i] - i + np.arange(n[i]) for i in nd])
        sd = w.sigma_d(pos_d.astype(np.float64), K[req_d])
        rows = logit_rows(seed, step, req_d, pos_d, w.V, w.dtype, w.sigma_t, sd)
        draft[at_d] = rows
        ids[at_d] = draft_ids(seed, step, req_d, pos_d, rows, w.V, w.dtype, temps[req_d])
    ii, jj = np.meshgrid(np.arange(bs, dtype=np.int32), np.arange(w.k_max + 1, dtype=np.int32),
                         indexing="ij")
    u = uniforms(seed, ST_UNIFORM, step, ii.ravel(), jj.ravel()).reshape(bs, w.k_max + 1)
    return {"target": target, "draft": draft, "draft_ids": ids, "uniforms": u, "temps": temps}


def bf16_to_f32(u16: np.ndarray) -> np.ndarray:
    return (u16.astype(np.uint32) << 16).view(np.float32)
