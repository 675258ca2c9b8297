"""GPU parity of the online calibration calls (sd_calibrate,
sd_calibrate_apply) against the oracle's calibration step.

The update is floating point: the GPU sums in fp32 within a warp and fp64
across warps, the oracle in fp64.  The bound below follows from that: each
term e = sigmoid(z) - label carries a few fp32 roundings (|e| <= 1, error
about 3e-7), a warp sum of at most 8 slots a thread and 5 shuffle levels adds
about 13 roundings relative to the sum of |terms|, and the stored parameter
one more rounding.  1e-5 * lr * (1 + max |c|) + 1e-6 * (1 + |param|) covers it
with room.
"""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import speculative_decoding_verification_sd_gb300 as sd  # noqa: E402


def _dev(a, dt):
    a = np.ascontiguousarray(a, dt)
    if a.size == 0:
        a = np.zeros(1, dt)
    return torch.from_numpy(a).cuda()


def _case(rng, bs, k_max):
    dl = rng.integers(0, k_max + 1, bs).astype(np.int32)
    nv = np.array([rng.integers(0, k + 1) for k in dl], np.int32)
    acc = np.array([rng.integers(0, n + 1) for n in nv], np.int32)
    conf = rng.normal(0.5, 2.0, int(dl.sum())).astype(np.float32)
    w0 = rng.normal(1.0, 0.3, k_max).astype(np.float32)
    b0 = rng.normal(0.0, 0.5, k_max).astype(np.float32)
    return dl, nv, acc, conf, w0, b0


def _gpu_update(conf, dl, nv, acc, k_max, lr, w0, b0):
    w, b = _dev(w0, np.float32), _dev(b0, np.float32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    sd.sd_calibrate(_dev(conf, np.float32), _dev(dl, np.int32), _dev(nv, np.int32),
                    _dev(acc, np.int32), len(dl), k_max, lr, w, b, err)
    torch.cuda.synchronize()
    return w.cpu().numpy(), b.cpu().numpy(), int(err.item())


def _check_update(conf, dl, nv, acc, k_max, lr, w0, b0):
    gw, gb, err = _gpu_update(conf, dl, nv, acc, k_max, lr, w0, b0)
    assert err == 0
    o = oracle.calibrate(conf, dl, nv, acc, k_max, lr, w0.astype(np.float64), b0.astype(np.float64))
    cmax = float(np.abs(conf).max()) if conf.size else 0.0
    for j in range(k_max):
        if o["count"][j] == 0:  # untouched, bit for bit
            assert gw[j] == w0[j] and gb[j] == b0[j]
            continue
        assert abs(gw[j] - o["w"][j]) <= 1e-5 * lr * (1 + cmax) + 1e-6 * (1 + abs(o["w"][j])), j
        assert abs(gb[j] - o["b"][j]) <= 1e-5 * lr + 1e-6 * (1 + abs(o["b"][j])), j


def test_calibration_update_matches_oracle():
    rng = np.random.default_rng(4242)
    for trial in range(60):
        k_max = int(rng.integers(1, 16))
        P = 1 << (k_max - 1).bit_length()  # pow2ceil(k_max)
        bs = int(rng.integers(1, 8192 // P + 1)) if trial % 4 == 0 else int(rng.integers(1, 60))
        dl, nv, acc, conf, w0, b0 = _case(rng, bs, k_max)
        _check_update(conf, dl, nv, acc, k_max, 0.5, w0, b0)


@pytest.mark.parametrize("bs,k_max", [(8192, 1), (4096, 2), (512, 15), (1, 15), (1, 1)])
def test_calibration_at_the_slot_limit(bs, k_max):
    rng = np.random.default_rng(bs * 16 + k_max + 7)
    dl, nv, acc, conf, w0, b0 = _case(rng, bs, k_max)
    _check_update(conf, dl, nv, acc, k_max, 0.25, w0, b0)


def test_calibration_is_deterministic_and_lr_zero_keeps_parameters():
    rng = np.random.default_rng(5)
    dl, nv, acc, conf, w0, b0 = _case(rng, 300, 7)
    a = _gpu_update(conf, dl, nv, acc, 7, 0.3, w0, b0)
    b = _gpu_update(conf, dl, nv, acc, 7, 0.3, w0, b0)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    z = _gpu_update(conf, dl, nv, acc, 7, 0.0, w0, b0)
    assert np.array_equal(z[0], w0) and np.array_equal(z[1], b0)


def test_calibrated_logits_and_the_closed_loop():
    rng = np.random.default_rng(11)
    k_max = 7
    dl, nv, acc, conf, w0, b0 = _case(rng, 200, k_max)
    off = np.concatenate([[0], np.cumsum(dl)])
    pos = np.concatenate([np.arange(k) for k in dl]).astype(np.int64)
    ref = w0.astype(np.float64)[pos] * conf.astype(np.float64) + b0.astype(np.float64)[pos]
    c_d = _dev(conf, np.float32)
    out = torch.full_like(c_d, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    sd.sd_calibrate_apply(c_d, _dev(dl, np.int32), len(dl), k_max, _dev(w0, np.float32),
                          _dev(b0, np.float32), out, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = out.cpu().numpy()[: len(conf)]
    np.testing.assert_allclose(got, ref, rtol=2.0 ** -23, atol=1e-37)
    # in place gives the same values
    sd.sd_calibrate_apply(c_d, _dev(dl, np.int32), len(dl), k_max, _dev(w0, np.float32),
                          _dev(b0, np.float32), c_d, err)
    torch.cuda.synchronize()
    assert np.array_equal(c_d.cpu().numpy()[: len(conf)], got)
    # the planner takes the calibrated logits: its plan equals the oracle's on them
    cost = (1.0 + 0.01 * np.arange(len(dl) + int(dl.sum()) + 2)).astype(np.float32)
    r = sd.plan(_dev(dl, np.int32), k_max, conf=c_d[: max(len(conf), 1)], cost=_dev(cost, np.float32),
                T=len(dl))
    o = oracle.plan(got, dl, k_max, cost, len(dl))
    torch.cuda.synchronize()
    if not o["near"]:
        assert int(r.B.item()) == o["B"]
        assert np.array_equal(r.slot_mask.cpu().numpy(), o["slot_mask"])
    assert off[-1] == len(conf)


def test_calibration_device_checks():
    rng = np.random.default_rng(3)
    k_max = 4
    dl, nv, acc, conf, w0, b0 = _case(rng, 40, k_max)
    dl[0], nv[0], acc[0] = 3, 2, 1  # slots 0 (accepted) and 1 (rejected) observed
    conf = rng.normal(0.5, 2.0, int(dl.sum())).astype(np.float32)
    bad = acc.copy()
    bad[0] = 3  # more accepted than verified
    w, b, err = _gpu_update(conf, dl, nv, bad, k_max, 0.5, w0, b0)
    assert err & sd.SD_DEV_ERR_OUTCOME and np.array_equal(w, w0) and np.array_equal(b, b0)
    dl2, nv2 = dl.copy(), nv.copy()
    dl2[1], nv2[1], acc2 = 0, 2, acc.copy()  # verified slots a request never drafted
    acc2[1] = 0
    conf2 = rng.normal(0.5, 2.0, int(dl2.sum())).astype(np.float32)
    w, b, err = _gpu_update(conf2, dl2, nv2, acc2, k_max, 0.5, w0, b0)
    assert err & sd.SD_DEV_ERR_OUTCOME and np.array_equal(w, w0)
    nan = conf.copy()
    nan[1] = np.nan  # request 0, slot 1: observed
    w, b, err = _gpu_update(nan, dl, nv, acc, k_max, 0.5, w0, b0)
    assert err & sd.SD_DEV_ERR_CONF and np.array_equal(w, w0)
    dl3 = dl.copy()
    dl3[2] = k_max + 1
    conf3 = rng.normal(0.5, 2.0, int(dl3.sum())).astype(np.float32)
    w, b, err = _gpu_update(conf3, dl3, nv, acc, k_max, 0.5, w0, b0)
    assert err & sd.SD_DEV_ERR_DRAFT_LENS and np.array_equal(w, w0)
    out = torch.full((max(len(conf3), 1),), 7.0, device="cuda")
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    sd.sd_calibrate_apply(_dev(conf3, np.float32), _dev(dl3, np.int32), len(dl3), k_max,
                          _dev(w0, np.float32), _dev(b0, np.float32), out, e)
    torch.cuda.synchronize()
    assert int(e.item()) & sd.SD_DEV_ERR_DRAFT_LENS
    assert bool((out == 7.0).all())
