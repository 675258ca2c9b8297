"""sd_verify_noalloc (the entry point on the library's static scratch) gives
the same results as sd_verify on a caller workspace, call after call.

This file is collected last: it must pass on its own and after every other
GPU test (which leave their own workspaces behind but never the static
scratch in a state this entry point relies on)."""
import numpy as np
import pytest

import sdsynth as S
from harness import oracle_plan

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import speculative_decoding_verification_sd_gb300 as sd  # noqa: E402


def _inputs(w, seed):
    dev = torch.device("cuda:0")
    pi = S.plan_inputs(w, seed, 0)
    cu = oracle_plan(pi, w.k_max)["cu_seqlens"]
    vi = S.verify_inputs(w, seed, 0, cu, pi["draft_lens"])
    bf = w.dtype == S.BF16
    conv = (lambda a: torch.from_numpy(a.view(np.int16))) if bf else torch.from_numpy
    t = dict(target=conv(vi["target"]).to(dev),
             draft=conv(vi["draft"]).to(dev) if len(vi["draft"]) else None,
             ids=torch.from_numpy(np.ascontiguousarray(vi["draft_ids"], np.int32)).to(dev),
             u=torch.from_numpy(vi["uniforms"]).to(dev), temps=torch.from_numpy(vi["temps"]).to(dev),
             cu=torch.from_numpy(cu).to(dev))
    if t["ids"].numel() == 0:
        t["ids"] = torch.zeros(1, dtype=torch.int32, device=dev)
    return t, (sd.SD_BF16 if bf else sd.SD_F32)


def _outputs(w):
    dev = torch.device("cuda:0")
    return (torch.full((w.bs,), -7, dtype=torch.int32, device=dev),
            torch.full((w.bs, w.k_max + 1), -7, dtype=torch.int32, device=dev),
            torch.zeros(1, dtype=torch.int32, device=dev))


def _both(w, t, dt, ws):
    acc1, out1, err1 = _outputs(w)
    sd.sd_verify(t["target"], t["draft"], dt, w.V, t["ids"], t["u"], t["temps"], t["cu"], w.bs,
                 w.k_max, acc1, out1, None, err1, ws, ws.numel())
    acc2, out2, err2 = _outputs(w)
    sd.sd_verify_noalloc(t["target"], t["draft"], dt, w.V, t["ids"], t["u"], t["temps"], t["cu"],
                         w.bs, w.k_max, acc2, out2, None, err2)
    torch.cuda.synchronize()
    assert int(err1.item()) == 0 and int(err2.item()) == 0
    assert torch.equal(acc1, acc2)
    assert torch.equal(out1, out2)


@pytest.mark.parametrize("name,bs,k_max,V,dtype", [
    ("small_bf16", 32, 5, 20000, S.BF16),
    ("small_f32_unaligned", 24, 7, 1003, S.F32),
    ("adaptive", 256, 7, 129280, S.BF16),
])
def test_noalloc_matches_workspace_entry_point_two_calls(name, bs, k_max, V, dtype):
    w = S.WORKLOADS["adaptive_hc"].with_(bs=bs, k_max=k_max, T=bs, V=V, dtype=dtype, name=name)
    t, dt = _inputs(w, 5)
    ws = sd.verify_workspace(w.bs, w.k_max, w.V, dt)
    for _ in range(2):  # two calls in a row on both entry points
        _both(w, t, dt, ws)


def test_noalloc_after_a_larger_batch():
    """The cleared part follows the layout of each call's (bs, k_max)."""
    big = S.WORKLOADS["adaptive_hc"].with_(bs=64, k_max=7, T=64, V=8192, name="big")
    small = S.WORKLOADS["adaptive_hc"].with_(bs=8, k_max=3, T=8, V=8192, name="small")
    for w in (big, small, big):
        t, dt = _inputs(w, 11)
        _both(w, t, dt, sd.verify_workspace(w.bs, w.k_max, w.V, dt))


def test_noalloc_rejects_a_batch_beyond_the_scratch():
    """Refused on the host before any launch (the tensors below are too small
    for the sizes named: no kernel may ever run on them)."""
    bs, k_max, V = 4096, 15, 1 << 20
    assert sd.sd_verify_workspace_bytes(bs, k_max, V, sd.SD_BF16) > sd.SD_NOALLOC_SCRATCH_BYTES
    dev = torch.device("cuda:0")
    x = torch.zeros(16, dtype=torch.int32, device=dev)
    with pytest.raises(sd.SdError) as ei:
        sd.sd_verify_noalloc(x, x, sd.SD_BF16, V, x, x, x, x, bs, k_max, x, x, None, x)
    assert ei.value.status == sd.SD_ERR_UNSUPPORTED
    assert "static scratch" in str(ei.value)
