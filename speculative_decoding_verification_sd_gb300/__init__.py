"""GB300-native verification step of speculative decoding with adaptive
verification.

Two stages, both hand-written sm_103a CUDA kernels behind the C ABI of
``include/sd.h`` (``libsdverify.so``):

  sd_plan       survival -> global top-B (or one K for the batch) -> budget
                argmax -> varlen compaction
  sd_verify     vocab-wide speculative rejection sampling on compacted logits
  sd_calibrate  one online step of the per-position acceptance model (and
                sd_calibrate_apply: the calibrated logits for the next plan)

This module is the Python binding: the ``sd_*`` functions mirror the C entry
points one to one (argument marshalling only; tensors are passed as device
pointers), and :func:`plan` / :func:`verify` allocate the outputs with torch
for convenience.  PyTorch provides device memory and streams, nothing else.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass
from typing import Optional

import torch

from . import _lib
from ._lib import (SD_NOALLOC_SCRATCH_BYTES, SD_BF16, SD_DEV_ERR_CONF, SD_DEV_ERR_COST, SD_DEV_ERR_CU_SEQLENS,  # noqa: F401
                   SD_DEV_ERR_DRAFT_ID, SD_DEV_ERR_DRAFT_LENS, SD_DEV_ERR_LOGITS, SD_DEV_ERR_OUTCOME,
                   SD_DEV_ERR_TEMP, SD_DEV_ERR_TIMEOUT, SD_DEV_ERR_UNIFORM, SD_ERR_CUDA,
                   SD_ERR_DEVICE_CHECK, SD_ERR_INVALID_ARG, SD_ERR_SHAPE, SD_ERR_UNSUPPORTED,
                   SD_F32, SD_MAX_K, SD_MAX_PLAN_SLOTS, SD_MAX_ROW_BYTES, SD_MAX_V, SD_MAX_VERIFY_BS,
                   SD_MODE_ADAPTIVE, SD_MODE_ALL_SLOTS, SD_MODE_UNIFORM_K, SD_OK,
                   SD_VERIFY_DRAFT_PADDED, SD_VERIFY_EARLY_EXIT, SD_VERIFY_TEST_STALL, SdError,
                   sd_launch_cfg)

__all__ = [
    "sd_plan", "sd_verify", "sd_verify_ex", "sd_verify_noalloc", "sd_plan_workspace_bytes",
    "sd_verify_workspace_bytes", "sd_verify_launch_info", "sd_calibrate", "sd_calibrate_apply",
    "plan", "verify", "PlanResult",
    "VerifyResult", "SdError", "build", "library_path", "verify_workspace",
]


def build(force: bool = False):
    from ._build import build as _b
    return _b(force=force)


def library_path():
    return _lib.LIB_PATH


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"expected a CUDA tensor, an int address or None, got {type(t)}")
    if not t.is_cuda:
        raise ValueError("tensor arguments must live on the GPU")
    if not t.is_contiguous():
        raise ValueError("tensor arguments must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dt(dt):
    if dt in (SD_F32, torch.float32):
        return SD_F32
    if dt in (SD_BF16, torch.bfloat16):
        return SD_BF16
    raise ValueError(f"unsupported logits dtype {dt}")


# ---------------------------------------------------------------------------
# C ABI mirror (same names and argument order as include/sd.h)


def sd_plan_workspace_bytes(bs: int, k_max: int) -> int:
    return _lib.load().sd_plan_workspace_bytes(bs, k_max)


def sd_verify_workspace_bytes(bs: int, k_max: int, V: int, dt) -> int:
    return _lib.load().sd_verify_workspace_bytes(int(bs), int(k_max), int(V), _dt(dt))


def sd_plan(conf_logits, budget_conf, budget_draft_lens, bs_budget, draft_lens, bs, k_max,
            cost_table, cost_len, T, mode, B_out, slot_mask, num_verified, cu_seqlens, err_flag,
            workspace=None, ws_bytes=0, stream=None):
    st = _lib.load().sd_plan(_ptr(conf_logits), _ptr(budget_conf), _ptr(budget_draft_lens),
                             int(bs_budget), _ptr(draft_lens), int(bs), int(k_max),
                             _ptr(cost_table), int(cost_len), int(T), int(mode), _ptr(B_out),
                             _ptr(slot_mask), _ptr(num_verified), _ptr(cu_seqlens),
                             _ptr(err_flag), _ptr(workspace), int(ws_bytes), _stream(stream))
    return _lib.check("sd_plan", st)


def sd_verify(target_logits, draft_logits, dt, V, draft_ids, uniforms, temps, cu_seqlens, bs,
              k_max, accepted_len, out_tokens, probs_out, err_flag, workspace, ws_bytes,
              stream=None):
    st = _lib.load().sd_verify(_ptr(target_logits), _ptr(draft_logits), _dt(dt), int(V),
                               _ptr(draft_ids), _ptr(uniforms), _ptr(temps), _ptr(cu_seqlens),
                               int(bs), int(k_max), _ptr(accepted_len), _ptr(out_tokens),
                               _ptr(probs_out), _ptr(err_flag), _ptr(workspace), int(ws_bytes),
                               _stream(stream))
    return _lib.check("sd_verify", st)


def sd_calibrate(conf_logits, draft_lens, num_verified, accepted_len, bs, k_max, lr, w, b,
                 err_flag, stream=None):
    st = _lib.load().sd_calibrate(_ptr(conf_logits), _ptr(draft_lens), _ptr(num_verified),
                                  _ptr(accepted_len), int(bs), int(k_max), float(lr), _ptr(w),
                                  _ptr(b), _ptr(err_flag), _stream(stream))
    return _lib.check("sd_calibrate", st)


def sd_calibrate_apply(conf_logits, draft_lens, bs, k_max, w, b, conf_out, err_flag, stream=None):
    st = _lib.load().sd_calibrate_apply(_ptr(conf_logits), _ptr(draft_lens), int(bs), int(k_max),
                                        _ptr(w), _ptr(b), _ptr(conf_out), _ptr(err_flag),
                                        _stream(stream))
    return _lib.check("sd_calibrate_apply", st)


def _cfg(cfg):
    """sd_launch_cfg from a dict with any of blocks, flags, wait_limit_us."""
    if cfg is None:
        return None
    if isinstance(cfg, sd_launch_cfg):
        return ctypes.byref(cfg)
    c = sd_launch_cfg(int(cfg.get("blocks", 0)), int(cfg.get("flags", 0)),
                      int(cfg.get("wait_limit_us", 0)), 0)
    return ctypes.byref(c)


def sd_verify_ex(target_logits, draft_logits, dt, V, draft_ids, uniforms, temps, cu_seqlens, bs,
                 k_max, accepted_len, out_tokens, probs_out, err_flag, workspace, ws_bytes,
                 cfg=None, stream=None):
    st = _lib.load().sd_verify_ex(_ptr(target_logits), _ptr(draft_logits), _dt(dt), int(V),
                                  _ptr(draft_ids), _ptr(uniforms), _ptr(temps), _ptr(cu_seqlens),
                                  int(bs), int(k_max), _ptr(accepted_len), _ptr(out_tokens),
                                  _ptr(probs_out), _ptr(err_flag), _ptr(workspace), int(ws_bytes),
                                  _cfg(cfg), _stream(stream))
    return _lib.check("sd_verify_ex", st)


def sd_verify_noalloc(target_logits, draft_logits, dt, V, draft_ids, uniforms, temps, cu_seqlens,
                      bs, k_max, accepted_len, out_tokens, probs_out, err_flag, stream=None):
    st = _lib.load().sd_verify_noalloc(_ptr(target_logits), _ptr(draft_logits), _dt(dt), int(V),
                                       _ptr(draft_ids), _ptr(uniforms), _ptr(temps),
                                       _ptr(cu_seqlens), int(bs), int(k_max), _ptr(accepted_len),
                                       _ptr(out_tokens), _ptr(probs_out), _ptr(err_flag),
                                       _stream(stream))
    return _lib.check("sd_verify_noalloc", st)


def sd_verify_launch_info(V, dt, bs, blocks=0, flags=0) -> dict:
    req = sd_launch_cfg(int(blocks), int(flags), 0, 0)
    out = sd_launch_cfg()
    threads, buffers = ctypes.c_int(0), ctypes.c_int(0)
    smem = ctypes.c_size_t(0)
    st = _lib.load().sd_verify_launch_info(int(V), _dt(dt), int(bs), ctypes.byref(req),
                                           ctypes.byref(out), ctypes.byref(threads),
                                           ctypes.byref(buffers), ctypes.byref(smem))
    _lib.check("sd_verify_launch_info", st)
    return {"blocks": out.blocks, "threads": threads.value, "buffers": buffers.value,
            "smem_bytes": smem.value}


def verify_workspace(bs: int, k_max: int, V: int, dt, device=None) -> torch.Tensor:
    """A zero-filled workspace for sd_verify (zero-filled once; calls keep it
    so).  torch's CUDA allocations are 256-byte aligned, as the call requires."""
    return torch.zeros(sd_verify_workspace_bytes(bs, k_max, V, dt), dtype=torch.uint8,
                       device=device or torch.device("cuda"))


# ---------------------------------------------------------------------------
# Convenience layer: allocate outputs with torch and call the C ABI.


@dataclass
class PlanResult:
    B: torch.Tensor             # [1] int32
    slot_mask: torch.Tensor     # [bs, k_max] uint8
    num_verified: torch.Tensor  # [bs] int32
    cu_seqlens: torch.Tensor    # [bs+1] int32
    err: torch.Tensor           # [1] int32


@dataclass
class VerifyResult:
    accepted_len: torch.Tensor  # [bs] int32
    out_tokens: torch.Tensor    # [bs, k_max+1] int32
    probs: Optional[torch.Tensor]  # [bs*k_max, 2] fp32 or None
    err: torch.Tensor           # [1] int32


def plan(draft_lens: torch.Tensor, k_max: int, conf: Optional[torch.Tensor] = None,
         cost: Optional[torch.Tensor] = None, T: int = 0, mode: int = SD_MODE_ADAPTIVE,
         budget_conf: Optional[torch.Tensor] = None,
         budget_draft_lens: Optional[torch.Tensor] = None, err: Optional[torch.Tensor] = None,
         stream=None) -> PlanResult:
    dev = draft_lens.device
    bs = draft_lens.numel()
    B = torch.empty(1, dtype=torch.int32, device=dev)
    mask = torch.empty((bs, max(k_max, 1)), dtype=torch.uint8, device=dev)
    nv = torch.empty(bs, dtype=torch.int32, device=dev)
    cu = torch.empty(bs + 1, dtype=torch.int32, device=dev)
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device=dev)
    bsb = 0 if budget_draft_lens is None else budget_draft_lens.numel()
    # an empty packed array is still a valid (unread) buffer for the C ABI
    if conf is not None and conf.numel() == 0:
        conf = torch.zeros(1, dtype=torch.float32, device=dev)
    if budget_conf is not None and budget_conf.numel() == 0:
        budget_conf = torch.zeros(1, dtype=torch.float32, device=dev)
    sd_plan(conf, budget_conf, budget_draft_lens, bsb, draft_lens, bs, k_max, cost,
            0 if cost is None else cost.numel(), T, mode, B, mask, nv, cu, err, None, 0, stream)
    return PlanResult(B, mask[:, :k_max], nv, cu, err)


def verify(target: torch.Tensor, draft: Optional[torch.Tensor], dt, V: int,
           draft_ids: torch.Tensor, uniforms: torch.Tensor, temps: torch.Tensor,
           cu_seqlens: torch.Tensor, k_max: int, probs: bool = False,
           err: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
           cfg=None, stream=None) -> VerifyResult:
    dev = target.device
    bs = cu_seqlens.numel() - 1
    acc = torch.empty(bs, dtype=torch.int32, device=dev)
    out = torch.empty((bs, k_max + 1), dtype=torch.int32, device=dev)
    pr = torch.full((max(bs * k_max, 1), 2), float("nan"), dtype=torch.float32, device=dev) if probs else None
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = verify_workspace(bs, k_max, V, dt, dev)
    sd_verify_ex(target, draft, dt, V, draft_ids, uniforms, temps, cu_seqlens, bs, k_max, acc,
                 out, pr, err, workspace, workspace.numel(), cfg=cfg, stream=stream)
    return VerifyResult(acc, out, pr, err)
