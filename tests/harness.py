"""Shared helpers of the parity tests: run one verification step through the
C ABI and through the oracle on the same seeded bytes, and compare them with
the near-boundary allowance (decisions the oracle flags as within 1e-5
relative of their boundary may differ; every other result must be identical).
"""
from __future__ import annotations

import json
import os
from dataclasses import dataclass, field
from pathlib import Path

import numpy as np

import oracle
import sdsynth as S

ROOT = Path(__file__).resolve().parent.parent
PROB_RTOL = 1e-5


@dataclass
class Tally:
    decisions: int = 0
    near_mismatches: int = 0
    plan_decisions: int = 0
    plan_near_mismatches: int = 0
    cases: list = field(default_factory=list)

    def dump(self):
        """Writes the tally to $SD_TALLY_DIR/parity_tally.json when that is set."""
        d = os.environ.get("SD_TALLY_DIR")
        if d and Path(d).is_dir():
            (Path(d) / "parity_tally.json").write_text(json.dumps(self.__dict__, indent=1))


TALLY = Tally()


def torch_dev():
    import torch
    return torch.device("cuda:0")


def logits_to_dev(a):
    """Raw logits (fp32 array or bf16 bit patterns as uint16) to the device."""
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(torch_dev())
    return torch.from_numpy(a).to(torch_dev())


def alloc_rows(rows_cap, V, dtype, filled):
    """Device logits buffer of the full capacity with the compacted rows at the front."""
    import torch
    tdt = torch.float32 if dtype == S.F32 else torch.int16
    buf = torch.empty((max(rows_cap, 1), V), dtype=tdt, device=torch_dev())
    if len(filled):
        buf[: len(filled)].copy_(logits_to_dev(filled))
    return buf


def gpu_plan(pi, k_max, err=None):
    import torch
    import speculative_decoding_verification_sd_gb300 as sd
    d = lambda a, t: None if a is None else torch.from_numpy(np.ascontiguousarray(a, t)).to(torch_dev())
    r = sd.plan(d(pi["draft_lens"], np.int32), k_max, conf=d(pi["conf"], np.float32),
                cost=d(pi["cost"], np.float32), T=pi["T"], mode=pi["mode"],
                budget_conf=d(pi["budget_conf"], np.float32),
                budget_draft_lens=d(pi["budget_draft_lens"], np.int32), err=err)
    torch.cuda.synchronize()
    return {"B": int(r.B.item()), "slot_mask": r.slot_mask.cpu().numpy(),
            "num_verified": r.num_verified.cpu().numpy(), "cu_seqlens": r.cu_seqlens.cpu().numpy(),
            "err": int(r.err.item())}


def oracle_plan(pi, k_max):
    return oracle.plan(pi["conf"], pi["draft_lens"], k_max, pi["cost"], pi["T"], pi["mode"],
                       budget_conf=pi["budget_conf"], budget_draft_lens=pi["budget_draft_lens"])


def compare_plan(g, o, what=""):
    """Exact unless the oracle flags the plan near a boundary."""
    same = (g["B"] == o["B"] and np.array_equal(g["slot_mask"], o["slot_mask"])
            and np.array_equal(g["num_verified"], o["num_verified"])
            and np.array_equal(g["cu_seqlens"], o["cu_seqlens"]))
    TALLY.plan_decisions += 1
    if not same:
        assert o["near"] != 0, f"plan mismatch away from any boundary {what}: gpu B={g['B']} oracle B={o['B']}"
        TALLY.plan_near_mismatches += 1
    return same


def padded_rows(rows, cu, k_max, fill):
    """Compacted draft rows (or ids) to the uncompacted layout: (i, j) at
    i*k_max + j, the rest `fill`."""
    bs = len(cu) - 1
    shape = (max(bs * k_max, 1),) + rows.shape[1:]
    out = np.full(shape, fill, dtype=rows.dtype)
    for i in range(bs):
        n = int(cu[i + 1] - cu[i] - 1)
        if n:
            out[i * k_max: i * k_max + n] = rows[cu[i] - i: cu[i] - i + n]
    return out


def gpu_verify(w, vi, cu, k_max, cfg=None, rows_cap=None, workspace=None, padded=False):
    """Runs the sampling stage through the C ABI with capacity-sized buffers.
    With ``padded`` the draft rows and ids are passed uncompacted (row of
    (i, j) at i*k_max + j, SD_VERIFY_DRAFT_PADDED); probabilities are mapped
    back to the compacted index."""
    import torch
    import speculative_decoding_verification_sd_gb300 as sd
    bs = len(cu) - 1
    rows_cap = rows_cap or bs * (k_max + 1)
    draft, ids_h = vi["draft"], vi["draft_ids"]
    cfg = dict(cfg or {})
    if padded:
        draft = padded_rows(draft, cu, k_max, 0) if len(draft) else draft
        ids_h = padded_rows(ids_h, cu, k_max, 0)
        cfg["flags"] = cfg.get("flags", 0) | sd.SD_VERIFY_DRAFT_PADDED
    tgt = alloc_rows(rows_cap, w.V, w.dtype, vi["target"])
    dft = alloc_rows(max(bs * k_max, 1), w.V, w.dtype, draft)
    ids = torch.zeros(max(bs * k_max, 1), dtype=torch.int32, device=torch_dev())
    if len(ids_h):
        ids[: len(ids_h)] = torch.from_numpy(np.ascontiguousarray(ids_h, np.int32)).to(torch_dev())
    u = torch.from_numpy(vi["uniforms"]).to(torch_dev())
    tp = torch.from_numpy(vi["temps"]).to(torch_dev())
    cu_d = torch.from_numpy(np.asarray(cu, np.int32)).to(torch_dev())
    dt = sd.SD_F32 if w.dtype == S.F32 else sd.SD_BF16
    acc = torch.empty(bs, dtype=torch.int32, device=torch_dev())
    out = torch.empty((bs, k_max + 1), dtype=torch.int32, device=torch_dev())
    probs = torch.full((max(bs * k_max, 1), 2), float("nan"), dtype=torch.float32, device=torch_dev())
    err = torch.zeros(1, dtype=torch.int32, device=torch_dev())
    ws = workspace if workspace is not None else sd.verify_workspace(bs, k_max, w.V, dt, torch_dev())
    sd.sd_verify_ex(tgt, dft, dt, w.V, ids, u, tp, cu_d, bs, k_max, acc, out, probs, err, ws,
                    ws.numel(), cfg=cfg)
    torch.cuda.synchronize()
    pr = probs.cpu().numpy()
    if padded:
        comp = np.full((max(int(cu[-1]) - bs, 1), 2), np.nan, np.float32)
        for i in range(bs):
            n = int(cu[i + 1] - cu[i] - 1)
            comp[cu[i] - i: cu[i] - i + n] = pr[i * k_max: i * k_max + n]
        pr = comp
    return {"accepted_len": acc.cpu().numpy(), "out_tokens": out.cpu().numpy(),
            "probs": pr, "err": int(err.item()),
            "target_dev": tgt, "draft_dev": dft, "workspace": ws}


def oracle_verify(w, vi, cu, k_max, requests=None):
    return oracle.verify(vi["target"], vi["draft"] if len(vi["draft"]) else None, w.dtype, w.V,
                         vi["draft_ids"], vi["uniforms"], vi["temps"], cu, k_max,
                         requests=requests)


def compare_verify(g, o, cu, k_max, requests=None, what=""):
    """Per request: identical accepted length and tokens unless the oracle
    flagged a near-boundary decision in that request.  Probabilities p(x),
    q(x) of every slot the oracle tested agree within 1e-5 relative."""
    bs = len(cu) - 1
    reqs = range(bs) if requests is None else requests
    near_mis = 0
    for i in reqs:
        same = (g["accepted_len"][i] == o["accepted_len"][i]
                and np.array_equal(g["out_tokens"][i], o["out_tokens"][i]))
        if not same:
            assert o["near"][i] != 0, (
                f"request {i} differs away from any boundary {what}: gpu a={g['accepted_len'][i]} "
                f"{g['out_tokens'][i]} oracle a={o['accepted_len'][i]} {o['out_tokens'][i]}")
            near_mis += 1
            TALLY.cases.append({"what": what, "request": int(i), "near_flags": int(o["near"][i]),
                                "gpu": [int(g["accepted_len"][i])] + [int(x) for x in g["out_tokens"][i]],
                                "oracle": [int(o["accepted_len"][i])] + [int(x) for x in o["out_tokens"][i]]})
    TALLY.decisions += o["decisions"]
    TALLY.near_mismatches += near_mis
    if g["probs"] is not None:
        nd = int(cu[-1]) - bs
        px_o, qx_o = o["px"][:nd], o["qx"][:nd]
        m = ~np.isnan(px_o)
        if requests is not None:
            sel = np.zeros(nd, bool)
            for i in requests:
                sel[cu[i] - i: cu[i + 1] - i - 1] = True
            m &= sel
        if m.any():
            gp = g["probs"][:nd, 0].astype(np.float64)
            gq = g["probs"][:nd, 1].astype(np.float64)
            rel_p = np.abs(gp[m] - px_o[m]) / np.maximum(px_o[m], 1e-30)
            rel_q = np.abs(gq[m] - qx_o[m]) / np.maximum(qx_o[m], 1e-30)
            # probabilities below fp32's normal range carry absolute, not relative, precision
            big = (px_o[m] > 1e-30) & (qx_o[m] > 1e-30)
            assert rel_p[big].max(initial=0) <= PROB_RTOL, f"p(x) rel err {rel_p.max()} {what}"
            assert rel_q[big].max(initial=0) <= PROB_RTOL, f"q(x) rel err {rel_q.max()} {what}"
    return near_mis


def check_properties(g, cu, k_max, V, draft_ids):
    """Invariants that hold at any size."""
    bs = len(cu) - 1
    n = np.diff(cu) - 1
    a = g["accepted_len"]
    out = g["out_tokens"]
    assert np.all((a >= 0) & (a <= n))
    for i in range(bs):
        ai = a[i]
        assert np.all(out[i, ai + 1:] == -1)
        assert 0 <= out[i, ai] < V
        d0 = cu[i] - i
        assert np.array_equal(out[i, :ai], draft_ids[d0: d0 + ai])
