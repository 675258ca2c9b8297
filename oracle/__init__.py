"""CPU oracle for one speculative-decoding verification step -- TEST INFRASTRUCTURE.

This package is the plain, slow, fp64 restatement of the method that the CUDA
path is checked against.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import it; the product package never does.

The arithmetic lives in ``sd_oracle.cpp`` (sequential C++17, fp64, no shared
code with the CUDA library).  This module only compiles it and marshals numpy
arrays through ctypes.

Pins: every function here is pinned against things fixed outside it:
``tests/test_oracle_pins.py`` (the pages' worked examples in tests/golden/,
brute force on tiny inputs, closed forms, statistical tests),
``tests/test_oracle_uniform_k.py`` (the uniform-K planning mode),
``tests/test_oracle_calibration.py`` (the calibration step: finite differences of
its loss, hand-built outcomes, recovery of a generating model) and
``tests/test_oracle_plan_properties.py`` (planner invariants over random inputs).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "sd_oracle.cpp"
_LIB = _HERE / "libsd_oracle.so"

F32, BF16 = 0, 1
MODE_ADAPTIVE, MODE_ALL_SLOTS, MODE_UNIFORM_K = 0, 1, 2
NEAR_TOPB, NEAR_BUDGET = 1, 2
NEAR_ACCEPT, NEAR_CDF, DEGENERATE_RESIDUAL = 1, 2, 4


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> Path:
    """Compile the oracle with the host C++ compiler (no CUDA involved)."""
    if force or not _LIB.exists() or _LIB.stat().st_mtime < _SRC.stat().st_mtime:
        tmp = _LIB.with_suffix(f".so.tmp{os.getpid()}")
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-ffp-contract=off",
               "-Wall", "-Wextra", "-o", str(tmp), str(_SRC)]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(str(_LIB))
        P = ctypes.c_void_p
        i32 = ctypes.c_int
        lib.oracle_survival.argtypes = [P, P, i32, P]
        lib.oracle_plan.argtypes = [P, P, i32, i32, P, P, i32, P, i32, i32, i32,
                                    P, P, P, P, P, P]
        lib.oracle_verify.argtypes = [P, P, i32, i32, P, P, P, P, i32, i32, P, i32,
                                      P, P, P, P, P, P]
        lib.oracle_softmax.argtypes = [P, i32, i32, ctypes.c_double, P]
        lib.oracle_calibrate.argtypes = [P, P, P, P, i32, i32, ctypes.c_double, P, P, P, P, P]
        for f in (lib.oracle_survival, lib.oracle_plan, lib.oracle_verify, lib.oracle_softmax,
                  lib.oracle_calibrate):
            f.restype = i32
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _check(rc, what):
    if rc != 0:
        raise OracleError(f"{what} returned {rc}")


def calibrate(conf, draft_lens, num_verified, accepted_len, k_max, lr, w, b):
    """One online-calibration step of the per-position logistic acceptance
    model a = sigmoid(w_j c + b_j) from one step's verification outcomes.
    Returns the updated w, b (fp64), the gradients and the observation counts."""
    dl = _c(draft_lens, np.int32)
    bs = len(dl)
    conf = _c(conf, np.float32)
    nv = _c(num_verified, np.int32)
    acc = _c(accepted_len, np.int32)
    w2 = np.array(w, np.float64, copy=True).reshape(k_max)
    b2 = np.array(b, np.float64, copy=True).reshape(k_max)
    gw = np.zeros(k_max, np.float64)
    gb = np.zeros(k_max, np.float64)
    cnt = np.zeros(k_max, np.int32)
    if conf is not None and conf.size == 0:
        conf = np.zeros(1, np.float32)
    _check(_load().oracle_calibrate(_ptr(conf), _ptr(dl), _ptr(nv), _ptr(acc), bs, k_max,
                                    float(lr), _ptr(w2), _ptr(b2), _ptr(gw), _ptr(gb), _ptr(cnt)),
           "oracle_calibrate")
    return {"w": w2, "b": b2, "grad_w": gw, "grad_b": gb, "count": cnt}


def survival(conf, draft_lens):
    """fp64 survival probabilities of the packed slots."""
    conf = _c(conf, np.float32)
    dl = _c(draft_lens, np.int32)
    out = np.zeros(int(dl.sum()), np.float64)
    _check(_load().oracle_survival(_ptr(conf), _ptr(dl), len(dl), _ptr(out)), "oracle_survival")
    return out


def plan(conf, draft_lens, k_max, cost=None, T=0, mode=MODE_ADAPTIVE,
         budget_conf=None, budget_draft_lens=None):
    """Planning stage.  Returns a dict with B, slot_mask, num_verified,
    cu_seqlens, obj (objective per B of the budget set; per K in uniform-K
    mode) and near flags.  In uniform-K mode B is the number of verified
    slots and K* = max(num_verified)."""
    dl = _c(draft_lens, np.int32)
    bs = len(dl)
    conf = _c(conf, np.float32)
    cost = _c(cost, np.float32)
    bconf = _c(budget_conf, np.float32)
    bdl = _c(budget_draft_lens, np.int32)
    B = np.zeros(1, np.int32)
    mask = np.zeros(bs * k_max, np.uint8)
    nv = np.zeros(bs, np.int32)
    cu = np.zeros(bs + 1, np.int32)
    near = np.zeros(1, np.int32)
    nobj = 1
    if mode == MODE_ADAPTIVE and cost is not None:
        nbud = int(bdl.sum()) if bdl is not None else int(dl.sum())
        nobj = max(1, min(nbud, len(cost) - 1 - T) + 1)
    elif mode == MODE_UNIFORM_K:
        nobj = int(dl.max()) + 1 if bs else 1
    obj = np.full(nobj, np.nan, np.float64)
    rc = _load().oracle_plan(_ptr(conf), _ptr(dl), bs, k_max, _ptr(bconf), _ptr(bdl),
                             0 if bdl is None else len(bdl), _ptr(cost),
                             0 if cost is None else len(cost), int(T), int(mode),
                             _ptr(B), _ptr(mask), _ptr(nv), _ptr(cu), _ptr(obj), _ptr(near))
    _check(rc, "oracle_plan")
    return {"B": int(B[0]), "slot_mask": mask.reshape(bs, k_max), "num_verified": nv,
            "cu_seqlens": cu, "obj": obj, "near": int(near[0])}


def verify(target, draft, dtype, V, draft_ids, uniforms, temps, cu_seqlens, k_max,
           requests=None):
    """Sampling stage for all requests (or the listed ones).

    ``target``/``draft`` are the compacted logits as raw arrays (float32, or
    uint16 bit patterns for bf16).  Returns accepted_len, out_tokens, px, qx,
    near flags per request and the number of decisions taken."""
    cu = _c(cu_seqlens, np.int32)
    bs = len(cu) - 1
    tgt = np.ascontiguousarray(target)
    dft = None if draft is None else np.ascontiguousarray(draft)
    ids = _c(draft_ids, np.int32)
    u = _c(uniforms, np.float32)
    tp = _c(temps, np.float32)
    req = None if requests is None else _c(requests, np.int32)
    acc = np.full(bs, -1, np.int32)
    out = np.full((bs, k_max + 1), -1, np.int32)
    nd = max(1, int(cu[-1]) - bs)
    px = np.full(nd, np.nan, np.float64)
    qx = np.full(nd, np.nan, np.float64)
    near = np.zeros(bs, np.int32)
    dec = np.zeros(1, np.int64)
    if ids is None or len(ids) == 0:
        ids = np.zeros(1, np.int32)
    rc = _load().oracle_verify(_ptr(tgt), _ptr(dft), int(dtype), int(V), _ptr(ids), _ptr(u),
                               _ptr(tp), _ptr(cu), bs, int(k_max), _ptr(req),
                               0 if req is None else len(req), _ptr(acc), _ptr(out),
                               _ptr(px), _ptr(qx), _ptr(near), _ptr(dec))
    _check(rc, "oracle_verify")
    return {"accepted_len": acc, "out_tokens": out, "px": px, "qx": qx, "near": near,
            "decisions": int(dec[0])}


def softmax(row, dtype, tau):
    """fp64 softmax of one raw logit row at temperature tau."""
    r = np.ascontiguousarray(row)
    out = np.zeros(r.shape[-1], np.float64)
    _check(_load().oracle_softmax(_ptr(r), int(dtype), r.shape[-1], float(tau), _ptr(out)),
           "oracle_softmax")
    return out
