"""CPU-side checks of the C-ABI library: it loads without a GPU, exports every
symbol include/sd.h declares, and rejects invalid arguments on the host
before touching CUDA."""
import ctypes
import re
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent


@pytest.fixture(scope="module")
def lib():
    import torch  # noqa: F401  (shares its CUDA runtime with the library)
    import speculative_decoding_verification_sd_gb300 as sd
    sd.build()
    return sd._lib.load()


def declared_symbols():
    text = (ROOT / "include" / "sd.h").read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(sd_[a-z_]+)\s*\(", text)
    return sorted(set(names))


def test_header_declarations_are_exported(lib):
    names = declared_symbols()
    assert "sd_plan" in names and "sd_verify" in names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/sd.h but not exported"
    import speculative_decoding_verification_sd_gb300 as sd
    assert sorted(sd._lib.EXPORTS) == names


def test_abi_version_and_status_strings(lib):
    import speculative_decoding_verification_sd_gb300 as sd
    assert lib.sd_abi_version() == 2
    for st in (0, -1, -2, -3, -4, -5):
        assert sd._lib.status_string(st)


def test_workspace_sizes(lib):
    import speculative_decoding_verification_sd_gb300 as sd
    assert sd.sd_plan_workspace_bytes(256, 7) == 0
    # at least a 32-byte statistics record per target and draft row, and the
    # per-warp chunk sums of up to two final draws per request
    rows = 256 * 8 + 256 * 7
    assert sd.sd_verify_workspace_bytes(256, 7, 129280, sd.SD_BF16) >= rows * 32 + 2 * 256 * 16 * 8
    assert sd.sd_verify_workspace_bytes(256, 7, 129280, sd.SD_F32) > \
        sd.sd_verify_workspace_bytes(256, 7, 129280, sd.SD_BF16)
    assert sd.sd_verify_workspace_bytes(0, 7, 1024, sd.SD_BF16) == 0


@pytest.mark.parametrize("bs,k_max,V,elem", [(256, 7, 129280, 2), (1024, 7, 129280, 2),
                                              (64, 3, 256000, 2), (12, 5, 1000, 4),
                                              (1, 1, 16, 4), (4096, 15, 1 << 20, 2)])
def test_workspace_layout_exact(lib, bs, k_max, V, elem):
    """The sampling workspace, part by part, each 256-byte aligned: a 32-byte
    statistics record per target and draft row; the 2^-56 fixed-point chunk
    sums of up to two final draws per request (sixteen streaming warps, each
    with ceil(slice / 3 KB) draw chunks of a slice of ceil(V * elem / 16)
    bytes rounded up to 16); then the counters that are zero between calls:
    a pair counter per target row, a decision word per request, the draw
    list and the split-draw part counters (two per request each), and eight
    control words.  The GPU tests locate the zero part from this layout."""
    import speculative_decoding_verification_sd_gb300 as sd
    al = lambda v: (v + 255) // 256 * 256
    rows_t, rows_d = bs * (k_max + 1), bs * k_max
    sl = (-(-V * elem // 16) + 15) // 16 * 16
    ncd = -(-sl // 3072)
    rs = al((rows_t + rows_d) * 32)
    zero = al(rs + 2 * bs * 16 * ncd * 8)
    st = al(zero + rows_t * 4)
    dl = al(st + bs * 4)
    dpc = al(dl + 2 * bs * 4)
    ctrl = al(dpc + 2 * bs * 4)
    total = al(ctrl + 8 * 4)
    dt = sd.SD_BF16 if elem == 2 else sd.SD_F32
    assert sd.sd_verify_workspace_bytes(bs, k_max, V, dt) == total


FAKE = 1 << 20  # a non-null address that is never dereferenced on these paths


def test_plan_rejects_bad_arguments_on_host(lib):
    import speculative_decoding_verification_sd_gb300 as sd
    P = FAKE

    def call(**kw):
        a = dict(conf_logits=P, budget_conf=None, budget_draft_lens=None, bs_budget=0,
                 draft_lens=P, bs=4, k_max=3, cost_table=P, cost_len=65, T=4, mode=0, B_out=P,
                 slot_mask=P, num_verified=P, cu_seqlens=P, err_flag=P, workspace=None,
                 ws_bytes=0, stream=0)
        a.update(kw)
        return lib.sd_plan(a["conf_logits"], a["budget_conf"], a["budget_draft_lens"],
                           a["bs_budget"], a["draft_lens"], a["bs"], a["k_max"], a["cost_table"],
                           a["cost_len"], a["T"], a["mode"], a["B_out"], a["slot_mask"],
                           a["num_verified"], a["cu_seqlens"], a["err_flag"], a["workspace"],
                           a["ws_bytes"], a["stream"])

    assert call(bs=0) == sd.SD_ERR_INVALID_ARG
    assert call(k_max=-1) == sd.SD_ERR_INVALID_ARG
    assert call(k_max=16) == sd.SD_ERR_UNSUPPORTED
    assert call(mode=7) == sd.SD_ERR_INVALID_ARG
    assert call(draft_lens=None) == sd.SD_ERR_INVALID_ARG
    assert call(err_flag=None) == sd.SD_ERR_INVALID_ARG
    assert call(conf_logits=None) == sd.SD_ERR_INVALID_ARG
    assert call(T=0) == sd.SD_ERR_INVALID_ARG
    assert call(T=65) == sd.SD_ERR_SHAPE
    assert call(bs=2048, k_max=7) == sd.SD_ERR_UNSUPPORTED
    assert call(budget_conf=P, budget_draft_lens=None) == sd.SD_ERR_INVALID_ARG
    # the uniform-K mode needs the same inputs as the adaptive one
    U = sd.SD_MODE_UNIFORM_K
    assert call(mode=U, conf_logits=None) == sd.SD_ERR_INVALID_ARG
    assert call(mode=U, cost_table=None) == sd.SD_ERR_INVALID_ARG
    assert call(mode=U, T=0) == sd.SD_ERR_INVALID_ARG
    assert call(mode=U, T=65) == sd.SD_ERR_SHAPE
    assert call(mode=U, bs=2048, k_max=7) == sd.SD_ERR_UNSUPPORTED
    assert call(mode=3) == sd.SD_ERR_INVALID_ARG


def test_verify_rejects_bad_arguments_on_host(lib):
    import speculative_decoding_verification_sd_gb300 as sd
    P = FAKE
    nb = sd.sd_verify_workspace_bytes(4, 3, 1024, sd.SD_BF16)

    def call(**kw):
        a = dict(t=P, d=P, dt=1, V=1024, ids=P, u=P, temps=P, cu=P, bs=4, k_max=3, acc=P, out=P,
                 probs=None, err=P, ws=P, nb=nb, stream=0)
        a.update(kw)
        return lib.sd_verify(a["t"], a["d"], a["dt"], a["V"], a["ids"], a["u"], a["temps"],
                             a["cu"], a["bs"], a["k_max"], a["acc"], a["out"], a["probs"],
                             a["err"], a["ws"], a["nb"], a["stream"])

    assert call(bs=0) == sd.SD_ERR_INVALID_ARG
    assert call(k_max=20) == sd.SD_ERR_UNSUPPORTED
    assert call(bs=5000) == sd.SD_ERR_UNSUPPORTED
    assert call(dt=9) == sd.SD_ERR_INVALID_ARG
    assert call(V=0) == sd.SD_ERR_INVALID_ARG
    assert call(V=(1 << 20) + 1) == sd.SD_ERR_UNSUPPORTED
    assert call(dt=0, V=(1 << 19) + 1) == sd.SD_ERR_UNSUPPORTED  # fp32 row over 2 MiB
    assert b"SD_MAX" in lib.sd_last_error_string()
    assert call(t=None) == sd.SD_ERR_INVALID_ARG
    assert call(acc=None) == sd.SD_ERR_INVALID_ARG
    assert call(out=None) == sd.SD_ERR_INVALID_ARG
    assert call(ws=None) == sd.SD_ERR_INVALID_ARG
    assert call(ws=P + 16) == sd.SD_ERR_INVALID_ARG  # workspace not 256-byte aligned
    assert call(nb=nb - 1) == sd.SD_ERR_SHAPE
    assert b"ws_bytes" in lib.sd_last_error_string()
    for bad in (sd.sd_launch_cfg(-1, 0, 0, 0), sd.sd_launch_cfg(0, 0x40, 0, 0),
                sd.sd_launch_cfg(0, 0, -1, 0), sd.sd_launch_cfg(0, 0, 0, 1)):
        assert lib.sd_verify_ex(P, P, 1, 1024, P, P, P, P, 4, 3, P, P, None, P, P, nb,
                                ctypes.byref(bad), 0) == sd.SD_ERR_INVALID_ARG
    # a refused call leaves its own reason, a later one resets it
    assert call(bs=0) == sd.SD_ERR_INVALID_ARG and b"bs=0" in lib.sd_last_error_string()


def test_calibration_rejects_bad_arguments_on_host(lib):
    """sd_calibrate / sd_calibrate_apply refuse bad arguments before any CUDA
    call; k_max = 0 is a no-op that returns before any launch."""
    import speculative_decoding_verification_sd_gb300 as sd
    P = FAKE

    def upd(**kw):
        a = dict(conf=P, dl=P, nv=P, acc=P, bs=4, k_max=3, lr=0.1, w=P, b=P, err=P)
        a.update(kw)
        return lib.sd_calibrate(a["conf"], a["dl"], a["nv"], a["acc"], a["bs"], a["k_max"],
                                a["lr"], a["w"], a["b"], a["err"], 0)

    def app(**kw):
        a = dict(conf=P, dl=P, bs=4, k_max=3, w=P, b=P, out=P, err=P)
        a.update(kw)
        return lib.sd_calibrate_apply(a["conf"], a["dl"], a["bs"], a["k_max"], a["w"], a["b"],
                                      a["out"], a["err"], 0)

    assert upd(bs=0) == sd.SD_ERR_INVALID_ARG
    assert upd(k_max=-1) == sd.SD_ERR_INVALID_ARG
    assert upd(k_max=16) == sd.SD_ERR_UNSUPPORTED
    assert upd(bs=2048, k_max=7) == sd.SD_ERR_UNSUPPORTED
    assert upd(lr=-0.5) == sd.SD_ERR_INVALID_ARG
    assert upd(lr=float("nan")) == sd.SD_ERR_INVALID_ARG
    assert upd(lr=float("inf")) == sd.SD_ERR_INVALID_ARG
    for k in ("dl", "nv", "acc", "err", "conf", "w", "b"):
        assert upd(**{k: None}) == sd.SD_ERR_INVALID_ARG, k
    assert upd(k_max=0, conf=None, w=None, b=None) == sd.SD_OK
    assert app(bs=0) == sd.SD_ERR_INVALID_ARG
    assert app(k_max=16) == sd.SD_ERR_UNSUPPORTED
    for k in ("dl", "err", "conf", "w", "b", "out"):
        assert app(**{k: None}) == sd.SD_ERR_INVALID_ARG, k
    assert app(k_max=0, conf=None, w=None, b=None, out=None) == sd.SD_OK


def test_noalloc_rejects_on_host(lib):
    """sd_verify_noalloc refuses bad sizes before any CUDA call."""
    import speculative_decoding_verification_sd_gb300 as sd
    P = FAKE

    def call(bs, k_max, V=1024):
        return lib.sd_verify_noalloc(P, P, 1, V, P, P, P, P, bs, k_max, P, P, None, P, 0)

    assert call(0, 3) == sd.SD_ERR_INVALID_ARG
    assert call(4, 16) == sd.SD_ERR_UNSUPPORTED
    assert b"no error" not in lib.sd_last_error_string()
    assert sd.sd_verify_workspace_bytes(4096, 15, 1 << 20, sd.SD_BF16) > sd.SD_NOALLOC_SCRATCH_BYTES
    assert call(4096, 15, 1 << 20) == sd.SD_ERR_UNSUPPORTED
    assert b"static scratch" in lib.sd_last_error_string()


def test_binding_refuses_host_tensors(lib):
    import torch
    import speculative_decoding_verification_sd_gb300 as sd
    with pytest.raises(ValueError):
        sd.sd_verify_workspace_bytes(1, 1, 16, sd.SD_F32) and sd._ptr(torch.zeros(3))


def test_product_path_does_not_import_the_oracle():
    pkg = ROOT / "speculative_decoding_verification_sd_gb300"
    for f in list(pkg.rglob("*.py")) + list(pkg.rglob("*.cu")) + list(pkg.rglob("*.cuh")) + list(pkg.rglob("*.h")):
        text = f.read_text()
        assert "import oracle" not in text and "from oracle" not in text, f
        assert "sd_oracle" not in text, f
