"""ctypes binding of libsdverify.so (include/sd.h).

Argument marshalling only: every step of the verification path runs in the
library's CUDA kernels.  Tensors are passed as device pointers; ``None`` is a
NULL pointer.  If the library has not been built the import of a binding
function fails loudly -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

PKG = Path(__file__).resolve().parent
LIB_PATH = PKG / "libsdverify.so"

SD_OK, SD_ERR_INVALID_ARG, SD_ERR_SHAPE, SD_ERR_UNSUPPORTED, SD_ERR_CUDA, SD_ERR_DEVICE_CHECK = (
    0, -1, -2, -3, -4, -5)
SD_F32, SD_BF16 = 0, 1
SD_MODE_ADAPTIVE, SD_MODE_ALL_SLOTS, SD_MODE_UNIFORM_K = 0, 1, 2

SD_DEV_ERR_DRAFT_LENS = 0x001
SD_DEV_ERR_CONF = 0x002
SD_DEV_ERR_COST = 0x004
SD_DEV_ERR_CU_SEQLENS = 0x008
SD_DEV_ERR_DRAFT_ID = 0x010
SD_DEV_ERR_TEMP = 0x020
SD_DEV_ERR_UNIFORM = 0x040
SD_DEV_ERR_LOGITS = 0x080
SD_DEV_ERR_TIMEOUT = 0x100
SD_DEV_ERR_OUTCOME = 0x200

SD_MAX_K = 15
SD_MAX_PLAN_SLOTS = 8192
SD_MAX_VERIFY_BS = 4096
SD_MAX_V = 1 << 20
SD_MAX_ROW_BYTES = 2 << 20

SD_VERIFY_EARLY_EXIT = 0x1
SD_VERIFY_DRAFT_PADDED = 0x2
SD_VERIFY_TEST_STALL = 0x100

# Every symbol include/sd.h declares.
EXPORTS = ("sd_plan_workspace_bytes", "sd_plan", "sd_verify_workspace_bytes", "sd_verify",
           "sd_verify_ex", "sd_verify_noalloc", "sd_verify_launch_info", "sd_calibrate",
           "sd_calibrate_apply", "sd_status_string", "sd_last_error_string", "sd_abi_version")
SD_NOALLOC_SCRATCH_BYTES = 16 << 20  # include/sd.h


class sd_launch_cfg(ctypes.Structure):
    _fields_ = [("blocks", ctypes.c_int), ("flags", ctypes.c_int),
                ("wait_limit_us", ctypes.c_int), ("reserved", ctypes.c_int)]


class SdError(RuntimeError):
    def __init__(self, fn, status, text):
        super().__init__(f"{fn} failed: {status} ({text})")
        self.status = status


_lib = None


def load(path: Path | None = None) -> ctypes.CDLL:
    """Load (once) and type the library.  Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    p = Path(path) if path else LIB_PATH
    if not p.exists():
        raise RuntimeError(
            f"{p} is missing: build it with __graft_entry__.build() (nvcc, sm_103a). "
            "There is no CPU fallback.")
    lib = ctypes.CDLL(str(p))
    P, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.sd_abi_version.restype = i32
    lib.sd_abi_version.argtypes = []
    lib.sd_status_string.restype = ctypes.c_char_p
    lib.sd_status_string.argtypes = [i32]
    lib.sd_last_error_string.restype = ctypes.c_char_p
    lib.sd_last_error_string.argtypes = []
    lib.sd_plan_workspace_bytes.restype = sz
    lib.sd_plan_workspace_bytes.argtypes = [i32, i32]
    lib.sd_verify_workspace_bytes.restype = sz
    lib.sd_verify_workspace_bytes.argtypes = [i32, i32, i32, i32]
    lib.sd_plan.restype = i32
    lib.sd_plan.argtypes = [P, P, P, i32, P, i32, i32, P, i32, i32, i32, P, P, P, P, P, P, sz, P]
    lib.sd_verify.restype = i32
    lib.sd_verify.argtypes = [P, P, i32, i32, P, P, P, P, i32, i32, P, P, P, P, P, sz, P]
    lib.sd_verify_ex.restype = i32
    lib.sd_verify_ex.argtypes = [P, P, i32, i32, P, P, P, P, i32, i32, P, P, P, P, P, sz,
                                 ctypes.POINTER(sd_launch_cfg), P]
    lib.sd_verify_noalloc.restype = i32
    lib.sd_verify_noalloc.argtypes = [P, P, i32, i32, P, P, P, P, i32, i32, P, P, P, P, P]
    lib.sd_calibrate.restype = i32
    lib.sd_calibrate.argtypes = [P, P, P, P, i32, i32, ctypes.c_float, P, P, P, P]
    lib.sd_calibrate_apply.restype = i32
    lib.sd_calibrate_apply.argtypes = [P, P, i32, i32, P, P, P, P, P]
    lib.sd_verify_launch_info.restype = i32
    lib.sd_verify_launch_info.argtypes = [i32, i32, i32, ctypes.POINTER(sd_launch_cfg),
                                          ctypes.POINTER(sd_launch_cfg), ctypes.POINTER(i32),
                                          ctypes.POINTER(i32), ctypes.POINTER(sz)]
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().sd_status_string(status).decode()


def check(fn: str, status: int) -> int:
    """Raises SdError for a status other than SD_OK, with the library's
    reason for it (every entry point records one for the calling thread)."""
    if status != SD_OK:
        text = status_string(status) + ": " + load().sd_last_error_string().decode()
        raise SdError(fn, status, text)
    return status
