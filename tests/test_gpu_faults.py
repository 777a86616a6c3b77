"""Failure paths, made on the host: no test here faults, traps or hangs the GPU.

- A workspace cap (option workspace_limit) turns a call that needs more device memory into
  ACF_ERR_NOMEM with a message. The context keeps working once the cap is lifted.
- Launch-failure injection (option inject_launch_error n) reports the n-th kernel launch from then
  on as failed. The launch itself ran normally. The call returns ACF_ERR_CUDA at once, and the
  next call gives exactly the histogram it gives without the fault. Each stage of acf_correlate is
  hit in turn: catalog preparation, pair kernels, fix-ups, merges and omega.
"""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.fixture(scope="module")
def cat():
    c = synth.catalogs(5000, 4000, 10, 30.0, seed=61)
    return c, tuple(map(_dev, (c.ra_d, c.dec_d, c.ra_r, c.dec_r)))


def test_workspace_limit_gives_nomem_and_recovers(acf, cat):
    c, (ra_d, dec_d, ra_r, dec_r) = cat
    lib = acf.load()
    ctx = acf.Context(0)
    try:
        ctx.set_option("workspace_limit", 1 << 16)  # far below what 5000 galaxies need
        out = torch.empty(720, dtype=torch.int64, device="cuda")
        rc = lib.acf_histogram(ctx.handle, ra_d.data_ptr(), dec_d.data_ptr(), c.n_d, None, None, 0, 0.25, 720,
                               out.data_ptr())
        assert rc == acf.ACF_ERR_NOMEM
        assert "workspace_limit" in acf.acf_last_error(ctx.handle)
        with pytest.raises(acf.AcfError):
            ctx.set_option("workspace_limit", -1)
        ctx.set_option("workspace_limit", 0)
        h = acf.as_uint64(ctx.histogram(ra_d, dec_d))
        torch.cuda.synchronize()
        assert int(h.sum()) == c.n_d ** 2
    finally:
        ctx.close()


def test_injected_launch_failures_return_an_error_and_leave_the_context_usable(acf, cat):
    c, (ra_d, dec_d, ra_r, dec_r) = cat
    lib = acf.load()
    ctx = acf.Context(0)
    try:
        ref = [acf.as_uint64(h).copy() for h in ctx.correlate(ra_d, dec_d, ra_r, dec_r, 0.25, 720)[:3]]
        torch.cuda.synchronize()
        before = ctx.info("kernel_launches")
        ctx.correlate(ra_d, dec_d, ra_r, dec_r, 0.25, 720)
        torch.cuda.synchronize()
        per_call = ctx.info("kernel_launches") - before
        assert per_call > 10
        outs = [torch.empty(720, dtype=torch.int64, device="cuda") for _ in range(3)]
        om = torch.empty(720, dtype=torch.float64, device="cuda")
        for n in range(1, per_call + 1):
            ctx.set_option("inject_launch_error", n)
            rc = lib.acf_correlate(ctx.handle, ra_d.data_ptr(), dec_d.data_ptr(), c.n_d, ra_r.data_ptr(),
                                   dec_r.data_ptr(), c.n_r, 0.25, 720, outs[0].data_ptr(), outs[1].data_ptr(),
                                   outs[2].data_ptr(), om.data_ptr())
            assert rc == acf.ACF_ERR_CUDA, n
            assert "injected" in acf.acf_last_error(ctx.handle)
            got = [acf.as_uint64(h) for h in ctx.correlate(ra_d, dec_d, ra_r, dec_r, 0.25, 720)[:3]]
            torch.cuda.synchronize()
            for g, r in zip(got, ref):
                assert np.array_equal(g, r), n
        # past the last launch of a call the injection does not fire within it
        ctx.set_option("inject_launch_error", per_call + 1)
        ctx.correlate(ra_d, dec_d, ra_r, dec_r, 0.25, 720)
        torch.cuda.synchronize()
        ctx.set_option("inject_launch_error", 0)
    finally:
        ctx.close()
